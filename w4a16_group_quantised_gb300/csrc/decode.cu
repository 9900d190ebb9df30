// decode.cu -- skinny-M (M <= 8) split-K W4A16 GEMM for sm_103a.
//
// "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP skinny
// decode", PR description: batch sizes M <= 5 go to a skinny split-K GEMM
// optimised for single-token decode, reading the same packed [N, K/8]
// weights as the prefill path.  The skinny GEMM is bound by the weight
// stream ("a memory-bound kernel", "Upstream sync 67/N ... (conflict)",
// section "Upstream's Python side is kept -- and it does NOT work here").
//
// Design (GB300-first, not the pages' RDNA kernel):
//  * A warp owns R blocks of 16 weight rows and a slice of K.  Each lane
//    streams 16 bytes (32 weights) of rows g and g+8 per 128-wide K step with
//    non-allocating 128-bit loads, D steps deep in a register ring.
//  * Weights are dequantised in registers (dq_word_i4) and multiplied on the
//    tensor cores with mma.sync m16n8k16 (fp32 accumulate): A = 16 weight rows
//    x 16 k, B = x^T (k x 8 batch columns, rows >= M are zero).  The k order
//    inside an MMA is a permutation of the word's nibbles; the x operand is
//    staged in shared memory in the same permutation, so the dot product is
//    the plain one.
//  * Split-K: KW warps of a CTA and S CTAs of a thread-block cluster take
//    disjoint K slices; partial sums meet in shared memory and are reduced
//    across the cluster through distributed shared memory, in a fixed order
//    (deterministic, no global workspace, no atomics).
//  * Programmatic dependent launch: the first weight steps are loaded before
//    the grid-dependency wait; x and out are touched only after it.
//    Weights, scales and zero points must therefore not be written by the
//    immediately preceding kernel if that kernel triggers early launch.
#include <cooperative_groups.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {

struct DecodeParams {
    const uint16_t *x;
    const int32_t *qw;
    const uint16_t *scales;
    const int32_t *qz;
    uint16_t *out;
    int M, N, K, G, ng;
    int RW, KW, S;
    int nblk;    // full 128-wide K blocks
    int ntail;   // trailing 32-wide K units (0..3)
    int xpitch;  // bytes per x row in shared memory
};

template <int DT>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    if (DT == 0) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

template <int R>
struct WStep {
    uint4 wa[R], wb[R];      // 4 words of rows g and g+8, per row block
    uint32_t sa[R], sb[R];   // scale bits
    uint32_t za[R], zb[R];   // zero-point words (asymmetric)
};

template <int DT>
__device__ __forceinline__ uint16_t f32_to_dt(float v) {
    if (DT == 0) {
        __half h = __float2half_rn(v);
        return *reinterpret_cast<uint16_t *>(&h);
    } else {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        return *reinterpret_cast<uint16_t *>(&h);
    }
}

// Multiply one word of rows g and g+8 (4 nibble pairs each) into acc.
template <int DT>
__device__ __forceinline__ void mac_word(float (&acc)[4], uint32_t wa, uint32_t wb, uint32_t zla,
                                         uint32_t zha, uint32_t s2a, uint32_t zlb, uint32_t zhb,
                                         uint32_t s2b, uint4 xv) {
    uint32_t oa[4], ob[4];
    dq_word_i4<DT>(wa, zla, zha, s2a, oa);
    dq_word_i4<DT>(wb, zlb, zhb, s2b, ob);
    mma_16816<DT>(acc, oa[0], ob[0], oa[1], ob[1], xv.x, xv.y);
    mma_16816<DT>(acc, oa[2], ob[2], oa[3], ob[3], xv.z, xv.w);
}

template <int DT, bool ASYM, int R, int D>
__global__ void __launch_bounds__(256) decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int RW = p.RW, KW = p.KW, S = p.S;
    const int rw = warp % RW, kw = warp / RW;
    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int tile = blockIdx.x / S;
    const int rows_cta = 16 * R * RW;
    const int K8 = p.K >> 3;

    grid_dependents_launch();

    // ---- K slices: CTA (cluster rank) and warp (kw) ranges of 128-wide blocks
    const int NS = S * KW;
    const int cta_b0 = (int)((long long)rank * p.nblk / S);
    const int cta_b1 = (int)((long long)(rank + 1) * p.nblk / S);
    const int slice = rank * KW + kw;
    const int sb = (int)((long long)slice * p.nblk / NS);
    const int se = (int)((long long)(slice + 1) * p.nblk / NS);
    const bool last_cta = (rank == S - 1);
    const bool tail_warp = (slice == NS - 1) && p.ntail > 0;
    const int nsteps = se - sb;

    // ---- rows of this warp
    int rowA[R];
    bool vA[R], vB[R];
#pragma unroll
    for (int rb = 0; rb < R; ++rb) {
        int n0 = tile * rows_cta + (rw * R + rb) * 16;
        rowA[rb] = n0 + g;
        vA[rb] = rowA[rb] < p.N;
        vB[rb] = rowA[rb] + 8 < p.N;
    }

    auto load_step = [&](WStep<R> &st, int blk) {
        const int grp = (blk * 128 + 32 * t) / p.G;
#pragma unroll
        for (int rb = 0; rb < R; ++rb) {
            const int ra = rowA[rb], rbw = ra + 8;
            const int32_t *wa = p.qw + (size_t)ra * K8 + blk * 16 + 4 * t;
            const int32_t *wb = p.qw + (size_t)rbw * K8 + blk * 16 + 4 * t;
            st.wa[rb] = vA[rb] ? ldg_stream_v4(wa) : make_uint4(0, 0, 0, 0);
            st.wb[rb] = vB[rb] ? ldg_stream_v4(wb) : make_uint4(0, 0, 0, 0);
            st.sa[rb] = vA[rb] ? (uint32_t)__ldg(p.scales + (size_t)ra * p.ng + grp) : 0u;
            st.sb[rb] = vB[rb] ? (uint32_t)__ldg(p.scales + (size_t)rbw * p.ng + grp) : 0u;
            if (ASYM) {
                const int zr = (ra - g) >> 3;  // first row of the block is a multiple of 16
                st.za[rb] = vA[rb] ? (uint32_t)__ldg(p.qz + (size_t)zr * p.ng + grp) : 0u;
                st.zb[rb] = vB[rb] ? (uint32_t)__ldg(p.qz + (size_t)(zr + 1) * p.ng + grp) : 0u;
            }
        }
    };

    WStep<R> ring[D];
#pragma unroll
    for (int d = 0; d < D - 1; ++d)
        if (d < nsteps) load_step(ring[d], sb + d);

    // ---- x slice of this CTA -> shared memory (permuted), after the
    //      grid-dependency wait (x may be produced by the previous kernel).
    float *red = reinterpret_cast<float *>(smem);
    const int red_floats = KW * RW * R * 16 * 8;
    unsigned char *xs = smem + red_floats * 4;
    grid_dependency_wait();
    {
        const int cnb = cta_b1 - cta_b0;
        const int nch = cnb * 16 + (last_cta ? p.ntail * 4 : 0);
        const int kbase = cta_b0 * 128;
        const int total = p.M * nch;
        for (int i = threadIdx.x; i < total; i += blockDim.x) {
            const int m = i / nch, c = i % nch;
            uint4 v = *reinterpret_cast<const uint4 *>(p.x + (size_t)m * p.K + kbase + 8 * c);
            int pos;
            if (c < cnb * 16) {
                const int b = c >> 4, cc = c & 15;
                pos = b * 16 + (cc & 3) * 4 + (cc >> 2);  // chunk 4t+w stored at 4w+t
            } else {
                pos = c;
            }
            uint4 o;
            o.x = __byte_perm(v.x, v.z, 0x5410);  // (x0, x4)
            o.y = __byte_perm(v.x, v.z, 0x7632);  // (x1, x5)
            o.z = __byte_perm(v.y, v.w, 0x5410);  // (x2, x6)
            o.w = __byte_perm(v.y, v.w, 0x7632);  // (x3, x7)
            *reinterpret_cast<uint4 *>(xs + (size_t)m * p.xpitch + pos * 16) = o;
        }
    }
    __syncthreads();

    float acc[R][4];
#pragma unroll
    for (int rb = 0; rb < R; ++rb) acc[rb][0] = acc[rb][1] = acc[rb][2] = acc[rb][3] = 0.f;

    const bool has_x = g < p.M;
    const unsigned char *xrow = xs + (size_t)g * p.xpitch;

    auto compute_step = [&](const WStep<R> &st, int blk) {
        const int lb = blk - cta_b0;
        uint4 xv[4];
#pragma unroll
        for (int w = 0; w < 4; ++w)
            xv[w] = has_x ? *reinterpret_cast<const uint4 *>(xrow + (lb * 16 + 4 * w + t) * 16)
                          : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int rb = 0; rb < R; ++rb) {
            uint32_t zA = 8u, zB = 8u;
            if (ASYM) {
                zA = (st.za[rb] >> (4 * g)) & 0xFu;
                zB = (st.zb[rb] >> (4 * g)) & 0xFu;
            }
            const uint32_t zla = zlo2<DT>(zA), zha = zhi2<DT>(zA), s2a = rep2(st.sa[rb]);
            const uint32_t zlb = zlo2<DT>(zB), zhb = zhi2<DT>(zB), s2b = rep2(st.sb[rb]);
            mac_word<DT>(acc[rb], st.wa[rb].x, st.wb[rb].x, zla, zha, s2a, zlb, zhb, s2b, xv[0]);
            mac_word<DT>(acc[rb], st.wa[rb].y, st.wb[rb].y, zla, zha, s2a, zlb, zhb, s2b, xv[1]);
            mac_word<DT>(acc[rb], st.wa[rb].z, st.wb[rb].z, zla, zha, s2a, zlb, zhb, s2b, xv[2]);
            mac_word<DT>(acc[rb], st.wa[rb].w, st.wb[rb].w, zla, zha, s2a, zlb, zhb, s2b, xv[3]);
        }
    };

    for (int s0 = 0; s0 < nsteps; s0 += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int s = s0 + d;
            if (s < nsteps) {
                if (s + D - 1 < nsteps) load_step(ring[(d + D - 1) % D], sb + s + D - 1);
                compute_step(ring[d], sb + s);
            }
        }
    }

    // ---- trailing 32-wide units (K % 128), taken by the last slice
    if (tail_warp) {
        const int cnb = cta_b1 - cta_b0;
        for (int u = 0; u < p.ntail; ++u) {
            const int k0 = p.nblk * 128 + 32 * u;
            const int grp = k0 / p.G;
            uint4 xv = has_x ? *reinterpret_cast<const uint4 *>(xrow + (cnb * 16 + 4 * u + t) * 16)
                             : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int rb = 0; rb < R; ++rb) {
                const int ra = rowA[rb], rbw = ra + 8;
                uint32_t wa = vA[rb] ? ldg_stream_u32(p.qw + (size_t)ra * K8 + k0 / 8 + t) : 0u;
                uint32_t wb = vB[rb] ? ldg_stream_u32(p.qw + (size_t)rbw * K8 + k0 / 8 + t) : 0u;
                uint32_t sa = vA[rb] ? (uint32_t)__ldg(p.scales + (size_t)ra * p.ng + grp) : 0u;
                uint32_t sbv = vB[rb] ? (uint32_t)__ldg(p.scales + (size_t)rbw * p.ng + grp) : 0u;
                uint32_t zA = 8u, zB = 8u;
                if (ASYM) {
                    const int zr = (ra - g) >> 3;
                    zA = vA[rb] ? ((uint32_t)__ldg(p.qz + (size_t)zr * p.ng + grp) >> (4 * g)) & 0xFu : 0u;
                    zB = vB[rb] ? ((uint32_t)__ldg(p.qz + (size_t)(zr + 1) * p.ng + grp) >> (4 * g)) & 0xFu
                                : 0u;
                }
                mac_word<DT>(acc[rb], wa, wb, zlo2<DT>(zA), zhi2<DT>(zA), rep2(sa), zlo2<DT>(zB),
                             zhi2<DT>(zB), rep2(sbv), xv);
            }
        }
    }

    // ---- partial sums -> shared memory: red[kw][row block][16][8]
#pragma unroll
    for (int rb = 0; rb < R; ++rb) {
        float *r = red + ((size_t)(kw * RW * R + rw * R + rb) * 16) * 8;
        r[g * 8 + 2 * t] = acc[rb][0];
        r[g * 8 + 2 * t + 1] = acc[rb][1];
        r[(g + 8) * 8 + 2 * t] = acc[rb][2];
        r[(g + 8) * 8 + 2 * t + 1] = acc[rb][3];
    }

    if (S > 1) {
        cg::this_cluster().sync();
    } else {
        __syncthreads();
    }

    // ---- reduce over KW warps and S cluster ranks; rank r writes its share
    {
        const int total = rows_cta * p.M;
        const int i0 = (int)((long long)rank * total / S);
        const int i1 = (int)((long long)(rank + 1) * total / S);
        for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
            const int m = i / rows_cta, row = i % rows_cta;
            const int n = tile * rows_cta + row;
            if (n >= p.N) continue;
            const int off = ((row >> 4) * 16 + (row & 15)) * 8 + m;
            float sum = 0.f;
            for (int s = 0; s < S; ++s) {
                const float *rs = (S > 1) ? cg::this_cluster().map_shared_rank(red, s) : red;
                for (int k = 0; k < KW; ++k) sum += rs[(size_t)k * RW * R * 128 + off];
            }
            p.out[(size_t)m * p.N + n] = f32_to_dt<DT>(sum);
        }
    }

    if (S > 1) cg::this_cluster().sync();  // keep shared memory alive for readers
}

// ------------------------------------------------------------------ host side
static int xpitch_bytes(const DecodeCfg &c, int K) {
    const int nblk = K / 128, ntail = (K % 128) / 32;
    const int max_cnb = (nblk + c.S - 1) / c.S;
    int bytes = max_cnb * 256 + ntail * 64;
    bytes = ((bytes + 127) / 128) * 128 + 64;  // odd multiple of 64: rows g, g+1 on different banks
    return bytes;
}

size_t decode_smem_bytes(const DecodeCfg &c, int M, int K) {
    const size_t red = (size_t)c.KW * c.RW * c.R * 16 * 8 * 4;
    return red + (size_t)M * xpitch_bytes(c, K);
}

bool decode_cfg_valid(const DecodeCfg &c, int M, int K) {
    if (c.R != 1 && c.R != 2) return false;
    if (c.D != 2 && c.D != 4) return false;
    if (c.RW < 1 || c.KW < 1 || c.RW * c.KW > 8) return false;
    if (c.S < 1 || c.S > 8) return false;
    if (decode_smem_bytes(c, M, K) > 200 * 1024) return false;
    return true;
}

DecodeCfg decode_pick_cfg(int M, int N, int K, int G, int sym, int dtype, int sm_count) {
    (void)G; (void)sym; (void)dtype;
    DecodeCfg c{1, 4, 4, 1, 1};
    const int nblk = K / 128;
    const int row_blocks = (N + 15) / 16;
    const int target_warps = sm_count * 16;
    int ks = (target_warps + row_blocks - 1) / row_blocks;
    if (ks > 16) ks = 16;
    if (ks > nblk) ks = nblk > 0 ? nblk : 1;
    if (ks < 1) ks = 1;
    c.KW = ks >= 2 ? 2 : 1;
    c.S = (ks + c.KW - 1) / c.KW;
    if (c.S > 8) c.S = 8;
    while (c.S * c.KW > (nblk > 0 ? nblk : 1) && (c.S > 1 || c.KW > 1)) {
        if (c.S > 1) --c.S; else --c.KW;
    }
    while (decode_smem_bytes(c, M, K) > 200 * 1024 && c.S < 8) ++c.S;
    return c;
}

template <int DT, bool ASYM, int R, int D>
static cudaError_t launch_t(const DecodeParams &p, const DecodeCfg &c, size_t smem,
                            cudaStream_t s, bool pdl, int grid) {
    auto kern = decode_kernel<DT, ASYM, R, D>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(32 * c.RW * c.KW, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (c.S > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = c.S;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int DT, bool ASYM>
static cudaError_t launch_rd(const DecodeParams &p, const DecodeCfg &c, size_t smem,
                             cudaStream_t s, bool pdl, int grid) {
    if (c.R == 1)
        return c.D == 2 ? launch_t<DT, ASYM, 1, 2>(p, c, smem, s, pdl, grid)
                        : launch_t<DT, ASYM, 1, 4>(p, c, smem, s, pdl, grid);
    return c.D == 2 ? launch_t<DT, ASYM, 2, 2>(p, c, smem, s, pdl, grid)
                    : launch_t<DT, ASYM, 2, 4>(p, c, smem, s, pdl, grid);
}

cudaError_t launch_decode(const GemmArgs &a, const DecodeCfg &c, const DeviceInfo &dev,
                          cudaStream_t s, bool pdl) {
    (void)dev;
    DecodeParams p;
    p.x = (const uint16_t *)a.x;
    p.qw = a.qweight;
    p.scales = (const uint16_t *)a.scales;
    p.qz = a.qzeros;
    p.out = (uint16_t *)a.out;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = a.G;
    p.ng = a.K / a.G;
    p.RW = c.RW;
    p.KW = c.KW;
    p.S = c.S;
    p.nblk = a.K / 128;
    p.ntail = (a.K % 128) / 32;
    p.xpitch = xpitch_bytes(c, a.K);
    const int rows_cta = 16 * c.R * c.RW;
    const int tiles = (a.N + rows_cta - 1) / rows_cta;
    const int grid = tiles * c.S;
    const size_t smem = decode_smem_bytes(c, a.M, a.K);
    const bool asym = a.qzeros != nullptr;
    if (a.dtype == 0)
        return asym ? launch_rd<0, true>(p, c, smem, s, pdl, grid)
                    : launch_rd<0, false>(p, c, smem, s, pdl, grid);
    return asym ? launch_rd<1, true>(p, c, smem, s, pdl, grid)
                : launch_rd<1, false>(p, c, smem, s, pdl, grid);
}

}  // namespace w4a16
