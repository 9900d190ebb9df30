// decode_warp.cu -- skinny-M (M <= 8) W4A16 GEMM with one weight stream per
// warp (sm_103a).
//
// Same operation and arithmetic as decode.cu ("[ROCm][Kernel] Add
// HybridW4A16LinearKernel: Triton prefill + HIP skinny decode", PR
// description: a skinny split-K GEMM for single-token decode over the packed
// [N, K/8] weights); this kernel is laid out for the weight stream alone:
//
//  * Work is cut into cells of 32 weight rows x NBK * 128 k.  The grid is
//    T row groups x S K-splits (S CTAs form a thread-block cluster, one CTA
//    per SM); a CTA owns a rectangle of whole row units (32 rows) and whole
//    K columns (NBK * 128 k), sized so that every SM streams nearly the same
//    number of bytes.  Inside the CTA the rectangle's cells, taken row unit
//    by row unit, are split into NW contiguous runs, one per warp.
//  * Every warp is its own TMA producer: its lane 0 keeps NSW cells of its
//    run in flight in the warp's private shared-memory ring (one 3-D tensor
//    copy of 32 rows x NBK blocks x 64 B per cell) and refills a slot as soon
//    as the warp has read it.  With 8 issuing warps per SM, copies are not
//    serialised behind a single issuing thread, and no warp waits for the
//    others to free a slot.
//  * Scales (and zero points) of the rectangle are staged once into shared
//    memory in the MMA's lane order, and x is staged permuted, as in
//    decode.cu; a lane dequantises 4 words (32 weights) of rows g and g+8 of
//    each 16-row block per 128-k block (dq_word_i4) and multiplies on the
//    tensor cores (mma.sync m16n8k16, fp32 accumulate).
//  * Reduction, in a fixed order (deterministic): each warp stores one fp32
//    partial per row unit it touched; after the loop the partials of a row
//    unit are added in warp order, then across the S CTAs of the cluster
//    through distributed shared memory in rank order.
//  * Programmatic dependent launch: weights, scales and zero points are read
//    before the grid-dependency wait; x and out only after it.
//  * Every mbarrier wait is bounded; on a timeout the status word is set and
//    the warp leaves its loop.
#include <cooperative_groups.h>
#include <cuda.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "skinny.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {

namespace {

constexpr int kUnitRows = 32;                    // rows per cell (two 16-row MMA blocks)
constexpr int kBlkK = 128;                       // k per block: 16 words = 64 B a row
constexpr int kBlkBytes = kUnitRows * 64;        // one block of one cell: 2 KB
constexpr int kMaxSeg = 4;                       // row units one warp may touch

struct WParams {
    const uint16_t *x;
    const uint16_t *scales;
    const int32_t *qz;
    uint16_t *out;
    int *status;
    DqConsts dq;          // dequantiser masks / magics, passed as data (see dequant.cuh)
    int M, N, K, ng, log2G;
    int U, T, S, C, KB;          // row units, row groups, K splits, K columns, 128-k blocks
    int NW, NSW;
    int xpitch;                  // bytes per x row in shared memory
    int gw_max;                  // groups per CTA K range (max over ranks)
    uint32_t off_meta, off_x, off_red, off_fin, off_bar;
};

}  // namespace

template <int DT, bool ASYM, int NBK>
__global__ void __launch_bounds__(256, 2) decode_warp_kernel(const __grid_constant__ CUtensorMap tmap,
                                                             const WParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int S = p.S, NW = p.NW, NSW = p.NSW, M = p.M;
    constexpr uint32_t kCellBytes = (uint32_t)NBK * kBlkBytes;
    constexpr int kES = ASYM ? 8 : 4;              // meta entry: {s2} or {s2, zl2}

    // ---- this CTA's rectangle
    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int tg = blockIdx.x / S;
    const int u0 = (int)((long long)tg * p.U / p.T);
    const int a = (int)((long long)(tg + 1) * p.U / p.T) - u0;
    const int col0 = (int)((long long)rank * p.C / S);
    const int c = (int)((long long)(rank + 1) * p.C / S) - col0;
    const int kb0 = col0 * NBK;
    const int nbk = min(c * NBK, p.KB - kb0);      // 128-k blocks of the K range
    const int gA = (kb0 * kBlkK) >> p.log2G;       // first group of the range
    const int GW = (nbk * kBlkK) >> p.log2G;       // groups of the range
    const int row0 = u0 * kUnitRows;
    const int rows = a * kUnitRows;
    const int ncells = a * c;
    const int w0 = (int)((long long)warp * ncells / NW);
    const int nmine = (int)((long long)(warp + 1) * ncells / NW) - w0;

    const uint32_t my_ring = sbase + (uint32_t)warp * NSW * kCellBytes;
    const uint32_t my_bar = sbase + p.off_bar + (uint32_t)warp * NSW * 8u;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_bar + NW * NSW * 8);

    grid_dependents_launch();

    auto issue = [&](int i) {   // lane 0: the warp's i-th cell into slot i % NSW
        const int cell = w0 + i;
        const int u = cell / c, col = cell - (cell / c) * c;
        const uint32_t slot = (uint32_t)(i % NSW);
        const uint32_t bar = my_bar + 8u * slot;
        mbar_arrive_expect_tx(bar, kCellBytes);
        tma_load_3d(my_ring + slot * kCellBytes, &tmap, bar, 0, (u0 + u) * kUnitRows, (col0 + col) * NBK);
    };

    if (tid == 0) *abort_flag = 0;
    if (lane == 0) {
        for (int s = 0; s < NSW; ++s) mbar_init(my_bar + 8u * s, 1);
        fence_mbar_init();
        for (int i = 0; i < min(NSW, nmine); ++i) issue(i);
    }

    // ---- scales (and zero points) of the rectangle -> meta[row][group]
    {
        const int nmeta = rows * GW;
        const int nthr = blockDim.x;
        for (int i0 = tid; i0 < nmeta; i0 += 8 * nthr) {
            uint32_t sv[8], zv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * nthr;
                sv[j] = 0u;
                zv[j] = 0x88888888u;
                if (i < nmeta) {
                    const int r = i / GW, gl = i - (i / GW) * GW;
                    const int n = row0 + r;
                    if (n < p.N) {
                        sv[j] = __ldg(p.scales + (size_t)n * p.ng + gA + gl);
                        if (ASYM) zv[j] = (uint32_t)__ldg(p.qz + (size_t)(n >> 3) * p.ng + gA + gl);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * nthr;
                if (i < nmeta) {
                    const int r = i / GW;
                    const uint32_t s2 = rep2(sv[j]);
                    if (ASYM) {
                        const int n = row0 + r;
                        const uint32_t zl2 = zlo2<DT>((zv[j] >> (4 * (n & 7))) & 0xFu);
                        *reinterpret_cast<uint2 *>(smem + p.off_meta + (size_t)i * 8) = make_uint2(s2, zl2);
                    } else {
                        *reinterpret_cast<uint32_t *>(smem + p.off_meta + (size_t)i * 4) = s2;
                    }
                }
            }
        }
    }

    // ---- x of the K range -> shared memory, permuted; zero for k >= K
    grid_dependency_wait();
    {
        unsigned char *xs = smem + p.off_x;
        const int nch = nbk * 16;                  // 16-byte chunks per row
        const int kbase = kb0 * kBlkK;
        for (int i = tid; i < M * nch; i += blockDim.x) {
            const int m = i / nch, cc0 = i - (i / nch) * nch;
            const int k = kbase + 8 * cc0;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (k < p.K) v = *reinterpret_cast<const uint4 *>(p.x + (size_t)m * p.K + k);
            const int b = cc0 >> 4, cc = cc0 & 15;
            const int pos = b * 16 + (cc & 3) * 4 + (cc >> 2);   // chunk 4t+w stored at 4w+t
            uint4 o;
            o.x = __byte_perm(v.x, v.z, 0x5410);  // (x0, x4)
            o.y = __byte_perm(v.x, v.z, 0x7632);  // (x1, x5)
            o.z = __byte_perm(v.y, v.w, 0x5410);  // (x2, x6)
            o.w = __byte_perm(v.y, v.w, 0x7632);  // (x3, x7)
            *reinterpret_cast<uint4 *>(xs + (size_t)m * p.xpitch + pos * 16) = o;
        }
    }
    __syncthreads();

    // ---- main loop over the warp's cells (four accumulator chains per 16-row block)
    float acc[2][4][4];
#pragma unroll
    for (int rb = 0; rb < 2; ++rb)
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[rb][c4][e] = 0.f;

    // Lanes whose batch column g is >= M read x row 0: their MMA output
    // columns are never stored.
    const unsigned char *xrow = smem + p.off_x + (g < M ? g : 0) * p.xpitch + t * 16;
    const uint32_t zl_sym = zlo2<DT>(8u), zh_sym = zhi2<DT>(8u);
    const DqConsts dc = p.dq;
    const int log2G = p.log2G;

    // Partial sums of a finished row unit -> red[warp][seg][row][m] (m < M).
    float *my_red = reinterpret_cast<float *>(smem + p.off_red) + (size_t)warp * kMaxSeg * kUnitRows * M;
    auto finish_segment = [&](int seg) {
        float *rs = my_red + (size_t)seg * kUnitRows * M;
#pragma unroll
        for (int rb = 0; rb < 2; ++rb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * rb + g + ((e & 2) ? 8 : 0), m = 2 * t + (e & 1);
                const float v = chain_sum(acc[rb], e);
                if (m < M && seg < kMaxSeg) rs[r * M + m] = v;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) acc[rb][c4][e] = 0.f;
            }
        }
    };

    int cur_u = -1, nseg = 0;
    for (int i = 0; i < nmine; ++i) {
        const int cell = w0 + i;
        const int u = cell / c, col = cell - (cell / c) * c;
        if (u != cur_u) {
            if (cur_u >= 0) finish_segment(nseg++);
            cur_u = u;
        }
        const uint32_t slot = (uint32_t)(i % NSW);
        if (!mbar_wait_bounded(my_bar + 8u * slot, (uint32_t)((i / NSW) & 1), p.status, abort_flag)) break;
        const unsigned char *cb = smem + (size_t)(warp * NSW + (int)slot) * kCellBytes + t * 16;
        // meta rows g, g+8, g+16, g+24 of this row unit
        const unsigned char *mrow = smem + p.off_meta + (size_t)((u * kUnitRows + g) * GW) * kES;
        const int mstep = 8 * GW * kES;
#pragma unroll
        for (int b = 0; b < NBK; ++b) {
            const int lb = col * NBK + b;          // block within the K range
            if (lb < nbk) {
                const unsigned char *xb = xrow + lb * 256;
                const uint4 xv[4] = {sh_v4(xb), sh_v4(xb + 64), sh_v4(xb + 128), sh_v4(xb + 192)};
                const int gofs = ((lb * kBlkK + 32 * t) >> log2G) * kES;
#pragma unroll
                for (int rb = 0; rb < 2; ++rb) {
                    const unsigned char *wrow = cb + b * kBlkBytes + (16 * rb + g) * 64;
                    const uint4 wa = sh_v4(wrow);
                    const uint4 wb = sh_v4(wrow + 8 * 64);
                    const unsigned char *ma = mrow + 2 * rb * mstep + gofs;
                    uint32_t s2a, s2b, zla = zl_sym, zlb = zl_sym, zha = zh_sym, zhb = zh_sym;
                    if (ASYM) {
                        const uint2 va = sh_v2(ma);
                        const uint2 vb = sh_v2(ma + mstep);
                        s2a = va.x; zla = va.y; zha = zhi_from_zlo<DT>(zla);
                        s2b = vb.x; zlb = vb.y; zhb = zhi_from_zlo<DT>(zlb);
                    } else {
                        s2a = sh_u32(ma);
                        s2b = sh_u32(ma + mstep);
                    }
                    mac_block<DT, 4>(acc[rb], dc, wa, wb, zla, zha, s2a, zlb, zhb, s2b, xv);
                }
            }
        }
        fence_proxy_async_smem();   // this warp's reads of the slot before the copy that refills it
        __syncwarp();
        if (lane == 0 && i + NSW < nmine) issue(i + NSW);
    }
    if (cur_u >= 0) finish_segment(nseg++);

    __syncthreads();

    // ---- add the warps' partials of each row unit, in warp order -> fin[row][m]
    float *fin = reinterpret_cast<float *>(smem + p.off_fin);
    for (int i = tid; i < rows * M; i += blockDim.x) {
        const int r = i / M, m = i - (i / M) * M;
        const int u = r / kUnitRows, rr = r - u * kUnitRows;
        float sum = 0.f;
        for (int ww = 0; ww < NW; ++ww) {
            const int a0 = (int)((long long)ww * ncells / NW);
            const int a1 = (int)((long long)(ww + 1) * ncells / NW);
            if (a1 > a0 && a0 < (u + 1) * c && a1 > u * c) {
                const int s = u - a0 / c;
                const float *red = reinterpret_cast<const float *>(smem + p.off_red) +
                                   ((size_t)ww * kMaxSeg + s) * kUnitRows * M;
                sum += red[rr * M + m];
            }
        }
        fin[r * 8 + m] = sum;
    }
    if (S > 1)
        cg::this_cluster().sync();
    else
        __syncthreads();

    // ---- add over the cluster's K splits, in rank order; rank r writes its share
    {
        const int total = rows * M;
        const int i0 = (int)((long long)rank * total / S);
        const int i1 = (int)((long long)(rank + 1) * total / S);
        for (int i = i0 + tid; i < i1; i += blockDim.x) {
            const int m = i / rows, r = i - (i / rows) * rows;
            const int n = row0 + r;
            if (n >= p.N) continue;
            float sum = 0.f;
            for (int s = 0; s < S; ++s) {
                const float *fs = (S > 1) ? cg::this_cluster().map_shared_rank(fin, s) : fin;
                sum += fs[r * 8 + m];
            }
            p.out[(size_t)m * p.N + n] = f32_to_dt<DT>(sum);
        }
    }
    if (S > 1) cg::this_cluster().sync();  // keep shared memory alive for the other ranks
}

// ------------------------------------------------------------------ host side
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Largest number of row units any warp of a CTA with a x c cells touches.
int max_segments(int a, int c, int NW) {
    const int ncells = a * c;
    int best = 0;
    for (int w = 0; w < NW; ++w) {
        const int w0 = (int)((long long)w * ncells / NW), w1 = (int)((long long)(w + 1) * ncells / NW);
        if (w1 > w0) best = std::max(best, (w1 - 1) / c - w0 / c + 1);
    }
    return best;
}

struct WLayout {
    uint32_t off_meta, off_x, off_red, off_fin, off_bar, total;
    int xpitch, gw_max;
};

WLayout wlayout(const DecodeWarpCfg &c, int M, int N, int K, int G, bool asym, int U, int T, int C) {
    (void)N;
    WLayout L;
    const int a_max = ceil_div(U, T);
    const int c_max = ceil_div(C, c.S);
    const int KB = ceil_div(K, kBlkK);
    const int nbk_max = std::min(c_max * c.NBK, KB);
    L.gw_max = nbk_max * kBlkK / G;
    uint32_t off = (uint32_t)c.NW * c.NSW * c.NBK * kBlkBytes;             // rings
    L.off_meta = off;
    off += (uint32_t)(a_max * kUnitRows) * L.gw_max * (asym ? 8 : 4);
    off = (off + 127u) & ~127u;
    L.off_x = off;
    int bytes = nbk_max * 256;
    L.xpitch = ((bytes + 127) / 128) * 128 + 64;   // odd multiple of 64: rows g, g+1 on other banks
    off += (uint32_t)M * L.xpitch;
    off = (off + 127u) & ~127u;
    L.off_red = off;                               // [NW][kMaxSeg][32 rows][M] fp32
    off += (uint32_t)c.NW * kMaxSeg * kUnitRows * M * 4;
    L.off_fin = off;
    off += (uint32_t)(a_max * kUnitRows) * 8 * 4;
    L.off_bar = off;
    off += (uint32_t)c.NW * c.NSW * 8 + 16;
    L.total = off + 1024;                          // slack to align the base to 1024
    return L;
}

}  // namespace

bool decode_warp_applicable(int M, int N, int K) {
    return M >= 1 && M <= 8 && K % kBlkK == 0 && N >= 8;
}

bool decode_warp_cfg_valid(const DecodeWarpCfg &c, int M, int N, int K, int G, bool asym, int sm_count,
                           int smem_optin) {
    if (!decode_warp_applicable(M, N, K)) return false;
    if (c.NBK != 1 && c.NBK != 2 && c.NBK != 4) return false;
    if (c.NW != 4 && c.NW != 8) return false;
    if (c.NSW < 1 || c.NSW > 8) return false;
    if (c.S < 1 || c.S > 8) return false;
    const int U = ceil_div(N, kUnitRows);
    const int KB = K / kBlkK;
    const int C = ceil_div(KB, c.NBK);
    if (c.S > C) return false;
    const int T = std::min(U, sm_count / c.S);
    if (T < 1) return false;
    for (int aa : {U / T, ceil_div(U, T)})
        for (int cc : {C / c.S, ceil_div(C, c.S)})
            if (aa > 0 && cc > 0 && max_segments(aa, cc, c.NW) > kMaxSeg) return false;
    const WLayout L = wlayout(c, M, N, K, G, asym, U, T, C);
    return (int)L.total <= smem_optin;
}

// Partition choice: the (NBK, S) that gives every SM the most even share of
// cells (ties: wider cells, then fewer K splits); 8 warps with 8 KB of ring
// each, so that a CTA of the next launch fits beside this one on the SM and
// starts streaming its weights early (programmatic dependent launch).
DecodeWarpCfg decode_warp_pick_cfg(int M, int N, int K, int G, int sym, int dtype, int sm_count, int smem_optin) {
    (void)dtype;
    DecodeWarpCfg best{0, 0, 0, 0};
    double best_eff = -1.0;
    const int U = ceil_div(N, kUnitRows);
    const int KB = K / kBlkK;
    for (int NBK : {2, 1}) {
        const int C = ceil_div(KB, NBK);
        for (int S = 1; S <= 8 && S <= C; ++S) {
            const int T = std::min(U, sm_count / S);
            if (T < 1) continue;
            const double cells = (double)ceil_div(U, T) * ceil_div(C, S);
            const double eff = ((double)U * C / sm_count) / cells * (NBK == 2 ? 1.0 : 0.97);
            for (int NW : {8, 4}) {
                DecodeWarpCfg c{NBK, S, NW, NBK == 1 ? 4 : 2};
                if (!decode_warp_cfg_valid(c, M, N, K, G, sym == 0, sm_count, smem_optin)) continue;
                if (eff > best_eff + 1e-9) {
                    best_eff = eff;
                    best = c;
                }
                break;
            }
        }
    }
    return best;   // NBK == 0: nothing fits
}

template <int DT, bool ASYM, int NBK>
static cudaError_t launch_w(const CUtensorMap &tm, const WParams &p, int S, int grid, int NW, size_t smem,
                            cudaStream_t s, bool pdl) {
    auto kern = decode_warp_kernel<DT, ASYM, NBK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (S > 1) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(32 * NW, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (S > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = S;
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
    return cudaLaunchKernelEx(&cfg, kern, tm, p);
}

template <int DT, bool ASYM>
static cudaError_t launch_w_nbk(int NBK, const CUtensorMap &tm, const WParams &p, int S, int grid, int NW,
                                size_t smem, cudaStream_t s, bool pdl) {
    switch (NBK) {
        case 1: return launch_w<DT, ASYM, 1>(tm, p, S, grid, NW, smem, s, pdl);
        case 2: return launch_w<DT, ASYM, 2>(tm, p, S, grid, NW, smem, s, pdl);
        default: return launch_w<DT, ASYM, 4>(tm, p, S, grid, NW, smem, s, pdl);
    }
}

cudaError_t launch_decode_warp(const GemmArgs &a, const DecodeWarpCfg &c, const DeviceInfo &dev, cudaStream_t s,
                               bool pdl) {
    if (dev.encode_tiled == nullptr) return cudaErrorNotSupported;
    const bool asym = a.qzeros != nullptr;
    const int U = ceil_div(a.N, kUnitRows);
    const int KB = a.K / kBlkK;
    const int C = ceil_div(KB, c.NBK);
    const int T = std::min(U, dev.sm_count / c.S);
    const WLayout L = wlayout(c, a.M, a.N, a.K, a.G, asym, U, T, C);

    // qweight [N, K/8] int32 seen as [K/128 blocks][N rows][16 words]: one
    // copy brings 32 rows x NBK blocks, each block row 64 contiguous bytes.
    CUtensorMap tm;
    {
        EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(dev.encode_tiled);
        cuuint64_t dims[3] = {16, (cuuint64_t)a.N, (cuuint64_t)KB};
        cuuint64_t strides[2] = {(cuuint64_t)(a.K / 8) * 4, 64};
        cuuint32_t box[3] = {16, (cuuint32_t)kUnitRows, (cuuint32_t)c.NBK};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, const_cast<int32_t *>(a.qweight), dims, strides,
                            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    WParams p;
    p.x = (const uint16_t *)a.x;
    p.scales = (const uint16_t *)a.scales;
    p.qz = a.qzeros;
    p.out = (uint16_t *)a.out;
    p.status = dev.status;
    p.dq = dq_consts_i4(a.dtype);
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.ng = a.K / a.G;
    p.log2G = a.G == 32 ? 5 : (a.G == 64 ? 6 : 7);
    p.U = U;
    p.T = T;
    p.S = c.S;
    p.C = C;
    p.KB = KB;
    p.NW = c.NW;
    p.NSW = c.NSW;
    p.xpitch = L.xpitch;
    p.gw_max = L.gw_max;
    p.off_meta = L.off_meta;
    p.off_x = L.off_x;
    p.off_red = L.off_red;
    p.off_fin = L.off_fin;
    p.off_bar = L.off_bar;
    const int grid = T * c.S;
    if (a.dtype == 0)
        return asym ? launch_w_nbk<0, true>(c.NBK, tm, p, c.S, grid, c.NW, L.total, s, pdl)
                    : launch_w_nbk<0, false>(c.NBK, tm, p, c.S, grid, c.NW, L.total, s, pdl);
    return asym ? launch_w_nbk<1, true>(c.NBK, tm, p, c.S, grid, c.NW, L.total, s, pdl)
                : launch_w_nbk<1, false>(c.NBK, tm, p, c.S, grid, c.NW, L.total, s, pdl);
}

}  // namespace w4a16
