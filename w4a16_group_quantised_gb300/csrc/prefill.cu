// prefill.cu -- fused-dequant W4A16 GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA, sm_103a).
//
// "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP skinny
// decode", PR description: batch sizes above the decode threshold go to a
// fused dequant GEMM (optimised for prefill / batched inference) that reads
// the same packed [N, K/8] weights.
//
// Design (GB300-first):
//  * One CTA computes a 128 (weight rows n) x BN (tokens m) output tile.  The
//    dequantised weights are the MMA's A operand (M = 128) and the
//    activations the B operand (N = BN <= 256), so the costly operand (W,
//    which must be dequantised by the SM's ALUs) is the smaller one per FLOP.
//  * Warp 0: TMA producer.  Per 64-wide K step it loads the x tile (BN rows x
//    128 B, 128-byte swizzle) and the packed weight tile (128 rows x 32 B)
//    into a `stages`-deep ring, completion tracked by transaction bytes.
//  * Warps 4..7: dequantisers (one weight row per thread).  They turn the
//    packed tile into a bf16/fp16 tile in the canonical K-major 128-byte
//    swizzled layout the tensor core reads, fence it into the async proxy and
//    arrive on the A-ring barrier.  Scales and zero points are prefetched
//    four steps ahead in registers.  After the main loop the same warps are
//    the epilogue: tcgen05.ld from TMEM, round once to the output dtype,
//    store (TMEM lane quadrant = warp % 4).
//  * Warp 1: TMEM allocation and the single-thread MMA issuer
//    (tcgen05.mma.cta_group::1.kind::f16, 128 x BN x 16 per instruction,
//    fp32 accumulator in TMEM); tcgen05.commit releases ring slots.
//  * Every mbarrier wait is bounded (%globaltimer); a wait that runs out sets
//    the device status word and a CTA abort flag, and every role leaves its
//    loop, so the CTA still frees its TMEM and exits.
#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"

#include <cuda.h>

namespace w4a16 {

constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBK = 64;           // K per pipeline step (one 128-byte swizzle row of 16-bit)
constexpr int kThreads = 256;
constexpr int kATileBytes = kBM * kBK * 2;   // 16 KB
constexpr int kWTileBytes = kBM * kBK / 2;   // 4 KB packed
constexpr int kScalePrefetch = 4;

struct PrefillParams {
    const uint16_t *scales;
    const int32_t *qz;
    uint16_t *out;
    int M, N, K, G, ng;
    int BN, stages, astages;
    int n_mtiles;
    int tmem_cols;
    int *status;
};

template <int DT>
__device__ __forceinline__ uint16_t f32_to_dt16(float v) {
    if (DT == 0) {
        __half h = __float2half_rn(v);
        return *reinterpret_cast<uint16_t *>(&h);
    } else {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        return *reinterpret_cast<uint16_t *>(&h);
    }
}

struct SmemLayout {
    uint32_t x_off, a_off, w_off, bar_off, total;
};

__host__ __device__ inline SmemLayout prefill_layout(int BN, int stages, int astages) {
    SmemLayout L;
    uint32_t off = 0;
    L.x_off = off;
    off += (uint32_t)stages * BN * 128;
    off = (off + 1023u) & ~1023u;
    L.a_off = off;
    off += (uint32_t)astages * kATileBytes;
    L.w_off = off;
    off += (uint32_t)stages * kWTileBytes;
    L.bar_off = off;
    off += (uint32_t)(2 * stages + 2 * astages + 1) * 8 + 16;
    L.total = off + 1024;  // slack for aligning the dynamic base to 1024
    return L;
}

template <int DT, bool ASYM>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_w, const PrefillParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const SmemLayout L = prefill_layout(p.BN, p.stages, p.astages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stages = p.stages, astages = p.astages;

    const int mt = blockIdx.x % p.n_mtiles;
    const int nt = blockIdx.x / p.n_mtiles;
    const int m0 = mt * p.BN, n0 = nt * kBM;
    const int nk = (p.K + kBK - 1) / kBK;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    const uint32_t bar_base = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (stages + s); };
    auto afull_bar = [&](int a) { return bar_base + 8u * (2 * stages + a); };
    auto aempty_bar = [&](int a) { return bar_base + 8u * (2 * stages + astages + a); };
    const uint32_t acc_bar = bar_base + 8u * (2 * stages + 2 * astages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.bar_off + 8 * (2 * stages + 2 * astages + 1));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t x_base = smem_u32(smem + L.x_off);
    const uint32_t a_base = smem_u32(smem + L.a_off);
    const uint32_t w_base = smem_u32(smem + L.w_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 128 + 1);
        }
        for (int a = 0; a < astages; ++a) {
            mbar_init(afull_bar(a), 128);
            mbar_init(aempty_bar(a), 1);
        }
        mbar_init(acc_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;

    grid_dependents_launch();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            grid_dependency_wait();  // x may be written by the previous kernel
            const uint32_t tx = (uint32_t)p.BN * 128u + (uint32_t)kWTileBytes;
            for (int i = 0; i < nk; ++i) {
                const int s = i % stages;
                const uint32_t ph = (uint32_t)((i / stages) & 1);
                if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, p.status, abort_flag)) break;
                mbar_arrive_expect_tx(full_bar(s), tx);
                tma_load_2d(x_base + (uint32_t)s * p.BN * 128u, &tmap_x, full_bar(s), i * kBK, m0);
                tma_load_2d(w_base + (uint32_t)s * kWTileBytes, &tmap_w, full_bar(s), i * (kBK / 8), n0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc_f16(DT, kBM, p.BN);
            for (int i = 0; i < nk; ++i) {
                const int s = i % stages, a = i % astages;
                if (!mbar_wait_bounded(full_bar(s), (uint32_t)((i / stages) & 1), p.status, abort_flag)) break;
                if (!mbar_wait_bounded(afull_bar(a), (uint32_t)((i / astages) & 1), p.status, abort_flag)) break;
                tc_fence_after();
                const uint32_t xa = x_base + (uint32_t)s * p.BN * 128u;
                const uint32_t aa = a_base + (uint32_t)a * kATileBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    tc_mma_f16(tmem_d, smem_desc_sw128(aa + kk * 32), smem_desc_sw128(xa + kk * 32),
                               idesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(empty_bar(s));
                tc_commit(aempty_bar(a));
            }
            tc_commit(acc_bar);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ dequantisers
        const int r = threadIdx.x - 128;          // weight row within the tile
        const int n = n0 + r;
        const bool vrow = n < p.N;
        const int zshift = 4 * (n & 7);
        // scale / zero-point register ring: [slot] = (lo-half group, hi-half group)
        uint32_t rs_lo[kScalePrefetch], rs_hi[kScalePrefetch], rz_lo[kScalePrefetch], rz_hi[kScalePrefetch];
        auto load_meta = [&](int i, uint32_t &slo, uint32_t &shi, uint32_t &zlo, uint32_t &zhi) {
            slo = shi = 0u;
            zlo = zhi = 0u;
            if (i < nk && vrow) {
                const int k_lo = i * kBK, k_hi = i * kBK + 32;
                const int g_lo = k_lo / p.G, g_hi = k_hi / p.G;
                slo = __ldg(p.scales + (size_t)n * p.ng + g_lo);
                if (ASYM) zlo = (uint32_t)__ldg(p.qz + (size_t)(n >> 3) * p.ng + g_lo);
                if (k_hi < p.K) {
                    shi = __ldg(p.scales + (size_t)n * p.ng + g_hi);
                    if (ASYM) zhi = (uint32_t)__ldg(p.qz + (size_t)(n >> 3) * p.ng + g_hi);
                }
            }
        };
#pragma unroll
        for (int d = 0; d < kScalePrefetch; ++d) load_meta(d, rs_lo[d], rs_hi[d], rz_lo[d], rz_hi[d]);

        const uint32_t a_row = (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
        const uint32_t sw = (uint32_t)(r & 7);
        bool ok = true;
        for (int i0 = 0; i0 < nk && ok; i0 += kScalePrefetch) {
#pragma unroll
            for (int d = 0; d < kScalePrefetch; ++d) {
                const int i = i0 + d;
                if (i < nk && ok) {
                    const uint32_t slo = rs_lo[d], shi = rs_hi[d];
                    uint32_t zlo = 8u, zhi = 8u;
                    if (ASYM) {
                        zlo = (rz_lo[d] >> zshift) & 0xFu;
                        zhi = (rz_hi[d] >> zshift) & 0xFu;
                    }
                    load_meta(i + kScalePrefetch, rs_lo[d], rs_hi[d], rz_lo[d], rz_hi[d]);

                    const int s = i % stages, a = i % astages;
                    if (!mbar_wait_bounded(full_bar(s), (uint32_t)((i / stages) & 1), p.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const unsigned char *wsrc = smem + L.w_off + (size_t)s * kWTileBytes + (size_t)r * 32;
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(wsrc);
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(wsrc + 16);
                    mbar_arrive(empty_bar(s));
                    if (!mbar_wait_bounded(aempty_bar(a), (uint32_t)((i / astages) & 1) ^ 1u, p.status,
                                           abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t zc_lo = zseq2<DT>(zlo), zc_hi = zseq2<DT>(zhi);
                    const uint32_t s2lo = rep2(slo), s2hi = rep2(shi);
                    unsigned char *adst = smem + L.a_off + (size_t)a * kATileBytes + a_row;
                    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[4];
                        dq_word_seq<DT>(words[c], c < 4 ? zc_lo : zc_hi, c < 4 ? s2lo : s2hi, o);
                        *reinterpret_cast<uint4 *>(adst + (((uint32_t)c ^ sw) << 4)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(afull_bar(a));
                }
            }
        }

        // ------------------------------------------------------------ epilogue
        if (ok && mbar_wait_bounded(acc_bar, 0u, p.status, abort_flag)) {
            tc_fence_after();
            const int q = warp & 3;
            const int nrow = n0 + 32 * q + lane;
            const uint32_t tbase = tmem_d + ((uint32_t)(32 * q) << 16);
            for (int c0 = 0; c0 < p.BN; c0 += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tbase + (uint32_t)c0, v);
                if (nrow < p.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m0 + c0 + j;
                        if (m < p.M) p.out[(size_t)m * p.N + nrow] = f32_to_dt16<DT>(__uint_as_float(v[j]));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_d, (uint32_t)p.tmem_cols);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PrefillCfg prefill_pick_cfg(int M, int N, int K, int G, int sym, int dtype, int sm_count) {
    (void)N; (void)K; (void)G; (void)sym; (void)dtype; (void)sm_count;
    PrefillCfg c;
    const int tiles_m = (M + 255) / 256;
    int bn = (M + tiles_m - 1) / tiles_m;
    bn = ((bn + 15) / 16) * 16;
    if (bn < 16) bn = 16;
    if (bn > 256) bn = 256;
    c.BN = bn;
    c.astages = 3;
    c.stages = 4;
    // keep within 227 KB: x ring dominates for large BN
    while (c.stages > 2 && prefill_layout(c.BN, c.stages, c.astages).total > 227 * 1024) --c.stages;
    return c;
}

template <int DT, bool ASYM>
static cudaError_t launch_t(const CUtensorMap &tx, const CUtensorMap &tw, const PrefillParams &p,
                            size_t smem, int grid, cudaStream_t s, bool pdl) {
    auto kern = prefill_kernel<DT, ASYM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1];
    int na = 0;
    if (pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, tx, tw, p);
}

cudaError_t prefill_prepare_device(const DeviceInfo &dev) {
    (void)dev;
    return cudaSuccess;
}

cudaError_t launch_prefill(const GemmArgs &a, const PrefillCfg &c, const DeviceInfo &dev,
                           cudaStream_t s, bool pdl) {
    if (dev.encode_tiled == nullptr) return cudaErrorNotSupported;
    EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(dev.encode_tiled);
    CUtensorMap tx, tw;
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)c.BN};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&tx, a.dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            2, const_cast<void *>(a.x), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)(a.K / 8), (cuuint64_t)a.N};
        cuuint64_t strides[1] = {(cuuint64_t)(a.K / 8) * 4};
        cuuint32_t box[2] = {(cuuint32_t)(kBK / 8), (cuuint32_t)kBM};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t *>(a.qweight), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    PrefillParams p;
    p.scales = (const uint16_t *)a.scales;
    p.qz = a.qzeros;
    p.out = (uint16_t *)a.out;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = a.G;
    p.ng = a.K / a.G;
    p.BN = c.BN;
    p.stages = c.stages;
    p.astages = c.astages;
    p.n_mtiles = (a.M + c.BN - 1) / c.BN;
    int cols = 32;
    while (cols < c.BN) cols <<= 1;
    p.tmem_cols = cols;
    p.status = dev.status;
    const int n_ntiles = (a.N + kBM - 1) / kBM;
    const int grid = n_ntiles * p.n_mtiles;
    const size_t smem = prefill_layout(c.BN, c.stages, c.astages).total;
    const bool asym = a.qzeros != nullptr;
    if (a.dtype == 0)
        return asym ? launch_t<0, true>(tx, tw, p, smem, grid, s, pdl)
                    : launch_t<0, false>(tx, tw, p, smem, grid, s, pdl);
    return asym ? launch_t<1, true>(tx, tw, p, smem, grid, s, pdl)
                : launch_t<1, false>(tx, tw, p, smem, grid, s, pdl);
}

}  // namespace w4a16
