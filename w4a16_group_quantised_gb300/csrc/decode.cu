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
//  * A CTA owns RT = 16 * R * NW weight rows and one K slice.  A producer
//    warp (warp NW, one thread) streams the slice's packed weights through
//    an NS-stage shared-memory ring with 2-D TMA boxes of RT rows x 128 k
//    (64 bytes a row, so a warp's 16-byte reads of rows g and g+1 fall on
//    disjoint banks); up to NS * NB boxes are in flight per CTA from the
//    first cycle, and the NW compute warps never issue or wait for a copy
//    on each other's behalf.  Scales and zero points of the slice are
//    staged once; x is staged permuted.
//  * Each warp owns R blocks of 16 rows.  Per 128-wide K step a lane takes
//    4 words (32 weights) of rows g and g+8, dequantises them in registers
//    (dq_word_i4) and multiplies on the tensor cores with mma.sync m16n8k16
//    (fp32 accumulate): A = 16 weight rows x 16 k, B = x^T (k x 8 batch
//    columns, rows >= M are zero).  The k order inside an MMA is a
//    permutation of each word's nibbles; x is staged in the same
//    permutation, so the dot product is the plain one.
//  * Split-K across the S CTAs of a thread-block cluster: ranks 1..S-1 send
//    their fp32 partials (real batch columns only) into rank 0's shared
//    memory with st.async, whose bytes complete rank 0's gather barrier, and
//    leave; rank 0 sums the S partials in rank order and stores y
//    (deterministic, no global workspace, no atomics, no cluster barrier at
//    the end).  A full ring stage arrives in one 3-D TMA copy when K is a
//    multiple of 128.
//  * Programmatic dependent launch: weights, scales and zero points are
//    requested before the grid-dependency wait; x and out are touched only
//    after it.  Weights, scales and zero points must therefore not be
//    written by the immediately preceding kernel if that kernel triggers
//    early launch.
//  * Fused epilogue: an optional bias [N] is added to the fp32 sums before
//    the one rounding; with SiLU-and-multiply (a merged gate/up weight of
//    N = 2 I rows, the gate rows first) a CTA's RT rows are RT / 2 gate rows
//    j0.. and the RT / 2 up rows I + j0.. (one TMA box over a [2][I] view of
//    the rows), and it writes silu(gate) * up for its RT / 2 outputs.
//  * Expert mode (the MoE grouped skinny GEMM): the weight is a stack of E
//    experts, [E * N] rows, and the grid runs over (token, expert slot) x
//    row tile x cluster rank; a CTA reads its slot's expert id (after the
//    grid-dependency wait: the routing may come from the previous kernel),
//    offsets its rows by e * N, multiplies that one token, and writes row
//    `slot` of the [T * topk, N] output, scaled by the slot's routing weight
//    when one is given.  An out-of-range id writes zeros and records
//    W4A16_ERR_ARG in the status word.
//  * Every mbarrier wait is bounded; on a timeout the status word is set and
//    the CTA leaves its loop.
#include <algorithm>
#include <mutex>
#include <cooperative_groups.h>
#include <cuda.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "skinny.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {

constexpr int kBoxK = 128;             // k per TMA box (16 int32 words = 64 B a row)
constexpr int kBoxRowBytes = kBoxK / 2;

struct DecodeParams {
    const uint16_t *x;
    const uint16_t *scales;
    const int32_t *qz;
    uint16_t *out;
    const uint16_t *bias;   // [N] or null
    int *status;
    DqConsts dq;          // dequantiser masks / magics, passed as data (see dequant.cuh)
    int M, N, K, G, ng, log2G;
    int NW, NB, NS, S;
    int nblk;        // K blocks of 128 (the last one may be partial)
    int wide;        // K % 128 == 0: full stages come in one copy (maps.wide)
    int xpitch;      // bytes per x row in shared memory
    int gmax;        // max groups per CTA slice
    int silu;        // SiLU-and-multiply epilogue: rows are [gate | up], I = N / 2 each
    int hold;        // test hook: issue no weight copies, so the bounded waits run out
#ifdef W4A16_DECODE_TRACE
    unsigned long long *trace;   // timeline hook: this launch's [kTraceCtas][kTraceEvents] stamps, or null
#endif
    // expert mode (expert_ids != null): x [T, K], out [T * topk, N], weights [E * N] rows
    const int *expert_ids;   // [T * topk]
    const float *route_w;    // [T * topk] or null
    int n_experts, topk, tiles;
};

// Weight tensor maps: `one` loads one 128-k block of RT rows (2-D, exact
// bounds); `wide` loads NB consecutive blocks in one copy (a 3-D view of the
// rows as [blocks][row][16 words], only when K is a multiple of 128, so that
// no block runs past the end of a row).  Fewer, larger copies per stage keep
// the producer thread's copy issue off the critical path.  With the SiLU
// epilogue both views gain a dimension of 2 (gate half, up half, I rows
// apart) and the boxes are RT / 2 rows high, so one copy still lands RT rows
// in the same [row][64 B] order.
struct DecodeMaps {
    CUtensorMap one;
    CUtensorMap wide;
};

struct DecodeSmem {
    uint32_t ring, meta, x, red, bars, total;
};

// meta: per (row, group) of the slice, {s2} (symmetric) or {s2, zl2}
// (asymmetric) -- the packed scale and low-magic zero constant, built once.
// red: the partial sums, [RT][8] fp32 without a K split; with one, the
// cluster's rank-0 CTA gathers every rank's partials there as [S][M][RT].
// bars: NS full and NS empty barriers, the abort flag, the gather barrier.
__host__ __device__ inline DecodeSmem decode_layout(int R, int NW, int NB, int NS, int M, int xpitch,
                                                    int gmax, bool asym, int S) {
    const int RT = 16 * R * NW;
    DecodeSmem L;
    uint32_t off = 0;
    L.ring = off;                                   // 128-B aligned for TMA
    off += (uint32_t)NS * NB * RT * kBoxRowBytes;
    L.meta = off;
    off += (uint32_t)RT * gmax * (asym ? 8 : 4);
    off = (off + 127u) & ~127u;
    L.x = off;                                      // [M][xpitch]
    off += (uint32_t)M * xpitch;
    L.red = off;
    off += (uint32_t)RT * 4 * (S > 1 && S * M > 8 ? S * M : 8);
    L.bars = off;
    off += (uint32_t)2 * NS * 8 + 24;
    L.total = off + 128;                            // slack to align the base to 128
    return L;
}

// Optional per-CTA timeline, compiled only into the trace build of the
// library (W4A16_DECODE_TRACE defined; the default build has none of it, so
// its kernel is unchanged).  The host hands a traced layer's launch (matched
// by N, K; up to four layers) its slice of the buffer that
// w4a16_debug_decode_trace installed, in the launch parameters.  Thread 0 of
// each of the first 512 CTAs writes %globaltimer at entry [0], when the
// grid-dependency wait returns [1], when x is staged [2], when its first
// weight stage is ready [3], at the end of its loop [4], when its cluster's
// partials are gathered [5, rank 0 only] and at exit [6]; [7] holds its
// cluster rank.
#ifdef W4A16_DECODE_TRACE
#define DECODE_STAMP(e) \
    do {                \
        if (trace) trace[e] = globaltimer(); \
    } while (0)
#else
#define DECODE_STAMP(e) \
    do {                \
    } while (0)
#endif

template <int DT, bool ASYM, int R, int NB>
__global__ void __launch_bounds__(288, 2) decode_kernel(const __grid_constant__ DecodeMaps maps,
                                                     const DecodeParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int NW = p.NW, NS = p.NS, S = p.S;
    const int RT = 16 * R * NW;
    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    int tile = blockIdx.x / S;
    const int silu = p.silu;
    const int RH = RT / 2;                           // SiLU: gate (and up) rows per CTA
    const int I = p.N / 2;
    const int M = p.M, K = p.K, gmax = p.gmax, log2G = p.log2G;
    // expert mode: this CTA's slot, its expert's first row, its token's x row and output row
    const uint16_t *xg = p.x;
    uint16_t *outg = p.out;
    int row_base = 0, slot = 0;
    bool bad_expert = false;
    if (p.expert_ids != nullptr) {
        slot = tile / p.tiles;
        tile -= slot * p.tiles;
        grid_dependency_wait();                      // the routing may be the previous kernel's output
        int e = p.expert_ids[slot];
        if (e < 0 || e >= p.n_experts) {
            bad_expert = true;
            e = 0;
            if (threadIdx.x == 0 && rank == 0) atomicExch(p.status, kStatusBadArg);
        }
        row_base = e * p.N;
        xg = p.x + (size_t)(slot / p.topk) * K;
        outg = p.out + (size_t)slot * p.N;
    }
    const int n_tile0 = silu ? tile * RH : tile * RT;
    const DecodeSmem L = decode_layout(R, NW, NB, NS, M, p.xpitch, gmax, ASYM, S);
#ifdef W4A16_DECODE_TRACE
    unsigned long long *trace = (p.trace != nullptr && threadIdx.x == 0 && blockIdx.x < kTraceCtas)
                                    ? p.trace + (size_t)blockIdx.x * kTraceEvents
                                    : nullptr;                 // thread 0 of a traced launch only
    if (trace) trace[7] = (unsigned long long)rank;
#endif
    DECODE_STAMP(0);

    grid_dependents_launch();

    // ---- K slice of this CTA, in 128-wide blocks
    const int b0 = (int)((long long)rank * p.nblk / S);
    const int b1 = (int)((long long)(rank + 1) * p.nblk / S);
    const int nb = bad_expert ? 0 : b1 - b0;
    const int nsteps = (nb + NB - 1) / NB;          // ring stages to consume
    const int g0 = (b0 * kBoxK) >> log2G;           // first group of the slice
    const int g1 = min(p.ng, (b1 * kBoxK + p.G - 1) >> log2G);
    const int ngs = bad_expert ? 0 : g1 - g0;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring = sbase + L.ring;
    const uint32_t stage_bytes = (uint32_t)NB * RT * kBoxRowBytes;
    const uint32_t bar0 = sbase + L.bars;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bars + 16 * NS);
    const uint32_t gbar = bar0 + 16u * NS + 8u;

    auto issue = [&](int step) {  // one thread: TMA all boxes of a ring stage
        const uint32_t sfull = bar0 + 8u * (uint32_t)(step % NS);
        const uint32_t sdst = ring + (uint32_t)(step % NS) * stage_bytes;
        const int bb = b0 + step * NB;
        const int nbox = min(NB, b1 - bb);
        mbar_arrive_expect_tx(sfull, (uint32_t)nbox * RT * kBoxRowBytes);
        if (p.wide && nbox == NB) {
            if (silu)
                tma_load_4d(sdst, &maps.wide, sfull, 0, n_tile0, 0, bb);
            else
                tma_load_3d(sdst, &maps.wide, sfull, 0, row_base + n_tile0, bb);
        } else {
            for (int j = 0; j < nbox; ++j) {
                const uint32_t d = sdst + (uint32_t)j * RT * kBoxRowBytes;
                if (silu)
                    tma_load_3d(d, &maps.one, sfull, (bb + j) * (kBoxK / 8), n_tile0, 0);
                else
                    tma_load_2d(d, &maps.one, sfull, (bb + j) * (kBoxK / 8), row_base + n_tile0);
            }
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar0 + 8u * s, 1);               // full
            mbar_init(bar0 + 8u * (NS + s), NW);       // empty: one arrive per compute warp
        }
        if (S > 1) mbar_init(gbar, 1);                // gather: rank 0's own arrive + the others' bytes
        *abort_flag = 0;
        fence_mbar_init();
        if (S > 1 && rank == 0) mbar_arrive_expect_tx(gbar, (uint32_t)(S - 1) * M * RT * 4u);
    }
    __syncthreads();
    if (S > 1) cluster_arrive_relaxed();   // rank 0's gather barrier is initialised

    float *red = reinterpret_cast<float *>(smem + L.red);
    if (warp == NW) {
        // ------------------------------------------------------------ producer
        // Step st refills slot st % NS once the compute warps have released
        // step st - NS from it.
        if (lane == 0 && !p.hold) {
            tma_prefetch_desc(&maps.one);
            if (p.wide) tma_prefetch_desc(&maps.wide);
            for (int st = 0; st < nsteps; ++st) {
                if (st >= NS &&
                    !mbar_wait_bounded(bar0 + 8u * (NS + st % NS), (uint32_t)((st / NS - 1) & 1), p.status,
                                       abort_flag))
                    break;
                issue(st);
            }
        }
        __syncwarp();
        grid_dependency_wait();   // before this warp joins the output stores
        if (S > 1) cluster_wait();
    } else {

        // ---- per-(row, group) constants of the slice (static: before the dependency wait).
        // RT is a power of two and the CTA has 2 / R threads per row; each thread
        // walks its row's groups with that stride, four loads in flight at a time.
        constexpr int kES = ASYM ? 8 : 4;                // meta entry: {s2} or {s2, zl2}
        const int nthr = 32 * NW;                        // compute threads
        {
            const int tpr = nthr / RT;
            const int r = (int)threadIdx.x & (RT - 1), gs = (int)threadIdx.x / RT;
            // weight row of tile row r (SiLU: gate rows j0.., then up rows I + j0..)
            const int n = silu ? (r < RH ? n_tile0 + r : I + n_tile0 + (r - RH)) : n_tile0 + r;
            const bool vr = silu ? (n_tile0 + (r < RH ? r : r - RH) < I) : n < p.N;
            const int nr = row_base + (vr ? n : 0);     // row in the (expert-stacked) weight
            const uint16_t *srow = p.scales + (size_t)nr * p.ng + g0;
            const int32_t *zrow = ASYM ? p.qz + (size_t)(nr >> 3) * p.ng + g0 : nullptr;
            const int zsh = 4 * (n & 7);
            unsigned char *mw = smem + L.meta + (size_t)r * gmax * kES;
            for (int gg0 = gs; gg0 < ngs; gg0 += 4 * tpr) {
                uint32_t sv[4], zv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int gg = gg0 + j * tpr;
                    sv[j] = 0u;
                    zv[j] = 0x88888888u;
                    if (vr && gg < ngs) {
                        sv[j] = __ldg(srow + gg);
                        if (ASYM) zv[j] = (uint32_t)__ldg(zrow + gg);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int gg = gg0 + j * tpr;
                    if (gg < ngs) {
                        if (ASYM)
                            *reinterpret_cast<uint2 *>(mw + gg * 8) =
                                make_uint2(rep2(sv[j]), zlo2<DT>((zv[j] >> zsh) & 0xFu));
                        else
                            *reinterpret_cast<uint32_t *>(mw + gg * 4) = rep2(sv[j]);
                    }
                }
            }
        }

        // ---- x slice -> shared memory, permuted; zero for k >= K
        grid_dependency_wait();
        DECODE_STAMP(1);
        {
            unsigned char *xs = smem + L.x;
            const int nch = nb * 16;                   // 16-byte chunks per row
            const int kbase = b0 * kBoxK;
            for (int i = threadIdx.x; i < M * nch; i += nthr) {
                const int m = i / nch, c = i - (i / nch) * nch;
                const int k = kbase + 8 * c;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (k < K) v = *reinterpret_cast<const uint4 *>(xg + (size_t)m * K + k);
                const int b = c >> 4, cc = c & 15;
                const int pos = b * 16 + (cc & 3) * 4 + (cc >> 2);   // chunk 4t+w stored at 4w+t
                uint4 o;
                o.x = __byte_perm(v.x, v.z, 0x5410);  // (x0, x4)
                o.y = __byte_perm(v.x, v.z, 0x7632);  // (x1, x5)
                o.z = __byte_perm(v.y, v.w, 0x5410);  // (x2, x6)
                o.w = __byte_perm(v.y, v.w, 0x7632);  // (x3, x7)
                *reinterpret_cast<uint4 *>(xs + (size_t)m * p.xpitch + pos * 16) = o;
            }
        }
        named_barrier_sync(1, (uint32_t)nthr);
        DECODE_STAMP(2);

        // Independent accumulator chains per row block: four for one block per
        // warp, two for two (keeps the register count, and so the CTAs per SM,
        // of the two-block form down).
        constexpr int NC = R == 1 ? 4 : 2;
        float acc[R][NC][4];
#pragma unroll
        for (int rb = 0; rb < R; ++rb)
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[rb][c][e] = 0.f;

        // Lanes whose batch column g is >= M read x row 0: their MMA output
        // columns are never stored, so no zeroing or predication is needed.
        const unsigned char *xrow = smem + L.x + (g < M ? g : 0) * p.xpitch + t * 16;
        const int rloc0 = warp * R * 16 + g;             // row of rb = 0 within the tile
        const unsigned char *mrow = smem + L.meta + rloc0 * gmax * kES;
        const uint32_t zl_sym = zlo2<DT>(8u), zh_sym = zhi2<DT>(8u);
        const DqConsts dc = p.dq;

        bool ok = true;
        int s = 0;                               // ring slot of this step
        uint32_t par = 0u;                       // its phase parity
        for (int step = 0; step < nsteps && ok; ++step) {
            if (!mbar_wait_bounded(bar0 + 8u * s, par, p.status, abort_flag)) {
                ok = false;
                break;
            }
            if (step == 0) DECODE_STAMP(3);
            const unsigned char *stage = smem + L.ring + (size_t)s * stage_bytes;
            const int lb0 = step * NB;
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int lb = lb0 + j;                   // slice-local block
                if (lb < nb) {
                    const int kb = (b0 + lb) * kBoxK;
                    const int gl = min(((kb + 32 * t) >> log2G) - g0, ngs - 1);
                    const unsigned char *xb = xrow + lb * 256;
                    const uint4 xv[4] = {sh_v4(xb), sh_v4(xb + 64), sh_v4(xb + 128), sh_v4(xb + 192)};
                    const unsigned char *box = stage + j * RT * kBoxRowBytes + t * 16 + rloc0 * kBoxRowBytes;
                    const unsigned char *mg = mrow + gl * kES;
#pragma unroll
                    for (int rb = 0; rb < R; ++rb) {
                        const uint4 wa = sh_v4(box + rb * 16 * kBoxRowBytes);
                        const uint4 wb = sh_v4(box + (rb * 16 + 8) * kBoxRowBytes);
                        const unsigned char *ma = mg + rb * 16 * gmax * kES;
                        uint32_t s2a, s2b, zla = zl_sym, zlb = zl_sym, zha = zh_sym, zhb = zh_sym;
                        if (ASYM) {
                            const uint2 va = sh_v2(ma);
                            const uint2 vb = sh_v2(ma + 8 * gmax * kES);
                            s2a = va.x; zla = va.y; zha = zhi_from_zlo<DT>(zla);
                            s2b = vb.x; zlb = vb.y; zhb = zhi_from_zlo<DT>(zlb);
                        } else {
                            s2a = sh_u32(ma);
                            s2b = sh_u32(ma + 8 * gmax * kES);
                        }
                        mac_block<DT, NC>(acc[rb], dc, wa, wb, zla, zha, s2a, zlb, zhb, s2b, xv);
                    }
                }
            }
            fence_proxy_async_smem();   // this warp's reads of the slot before the copy that refills it
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8u * (NS + s));
            if (++s == NS) {
                s = 0;
                par ^= 1u;
            }
        }

        DECODE_STAMP(4);
        // ---- partial sums -> shared memory: red[row][m]
        if (S == 1) {
#pragma unroll
            for (int rb = 0; rb < R; ++rb) {
                const int r0 = (warp * R + rb) * 16;
                red[(r0 + g) * 8 + 2 * t] = chain_sum(acc[rb], 0);
                red[(r0 + g) * 8 + 2 * t + 1] = chain_sum(acc[rb], 1);
                red[(r0 + g + 8) * 8 + 2 * t] = chain_sum(acc[rb], 2);
                red[(r0 + g + 8) * 8 + 2 * t + 1] = chain_sum(acc[rb], 3);
            }
        } else {
            // partials of the real batch columns into slot `rank` of rank 0's
            // gather buffer, [S][M][RT]: rank 0 plainly, the others with
            // asynchronous stores counted by rank 0's gather barrier
            cluster_wait();
            const uint32_t gbase = mapa_shared(smem_u32(red), 0u) + (uint32_t)rank * M * RT * 4u;
            const uint32_t gbar0 = mapa_shared(gbar, 0u);
#pragma unroll
            for (int rb = 0; rb < R; ++rb) {
                const int r0 = (warp * R + rb) * 16;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = r0 + g + (e >= 2 ? 8 : 0), col = 2 * t + (e & 1);
                    if (col < M) {
                        if (rank == 0)
                            red[col * RT + row] = chain_sum(acc[rb], e);
                        else
                            st_async_f32(gbase + (uint32_t)(col * RT + row) * 4u, chain_sum(acc[rb], e), gbar0);
                    }
                }
            }
        }
    }

    // the fp32 sum of tile row `row`, batch column m, over the cluster's ranks
    // in rank order (S > 1: rank 0's gather buffer [S][M][RT]), plus the bias
    auto row_sum = [&](int m, int row, int n) -> float {
        float sum;
        if (S == 1) {
            sum = red[row * 8 + m];
        } else {
            sum = red[m * RT + row];
            for (int q = 1; q < S; ++q) sum += red[(q * M + m) * RT + row];
        }
        if (p.bias != nullptr) sum += dt_to_f32<DT>(p.bias[n]);
        return sum;
    };
    if (S == 1 || rank == 0) {
        // rank 0 of a cluster: own partials (this CTA) and the other ranks'
        // (their bytes complete the gather barrier)
        __syncthreads();
        if (S > 1) mbar_wait_cluster_bounded(gbar, 0u, p.status, abort_flag);
        DECODE_STAMP(5);
        if (!silu) {
            const float rw = p.route_w != nullptr ? p.route_w[slot] : 1.0f;
            for (int i = threadIdx.x; i < RT * M; i += blockDim.x) {
                const int m = i / RT, row = i - (i / RT) * RT;
                const int n = n_tile0 + row;
                if (n < p.N) outg[(size_t)m * p.N + n] = f32_to_dt<DT>(row_sum(m, row, n) * rw);
            }
        } else {
            for (int i = threadIdx.x; i < RH * M; i += blockDim.x) {
                const int m = i / RH, row = i - (i / RH) * RH;
                const int j = n_tile0 + row;
                if (j >= I) continue;
                const float gte = row_sum(m, row, j), up = row_sum(m, RH + row, I + j);
                p.out[(size_t)m * I + j] = f32_to_dt<DT>(gte / (1.0f + expf(-gte)) * up);
            }
        }
    }
    DECODE_STAMP(6);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static int decode_gmax(const DecodeCfg &c, int K, int G) {
    const int nblk = (K + kBoxK - 1) / kBoxK;
    const int max_nb = (nblk + c.S - 1) / c.S;
    return (max_nb * kBoxK) / G + 2;
}

static int decode_xpitch(const DecodeCfg &c, int K) {
    const int nblk = (K + kBoxK - 1) / kBoxK;
    const int max_nb = (nblk + c.S - 1) / c.S;
    int bytes = max_nb * 256;
    bytes = ((bytes + 127) / 128) * 128 + 64;  // odd multiple of 64: rows g, g+1 on other banks
    return bytes;
}

size_t decode_smem_bytes(const DecodeCfg &c, int M, int K, int G, bool asym) {
    return decode_layout(c.R, c.NW, c.NB, c.NS, M, decode_xpitch(c, K), decode_gmax(c, K, G), asym, c.S).total;
}

bool decode_cfg_valid(const DecodeCfg &c, int M, int K, int G, bool asym) {
    if (c.R != 1 && c.R != 2) return false;
    if (c.NW != 1 && c.NW != 2 && c.NW != 4 && c.NW != 8) return false;
    if (c.NB != 1 && c.NB != 2 && c.NB != 4) return false;
    if (c.NS < 2 || c.NS > 8) return false;
    if (c.S < 1 || c.S > 8) return false;
    if (16 * c.R * c.NW > 256) return false;        // TMA box height limit
    if (decode_smem_bytes(c, M, K, G, asym) > 220 * 1024) return false;
    return true;
}

template <int DT, bool ASYM, int R, int NB>
static cudaError_t launch_t(const DecodeMaps &tw, const DecodeParams &p, const DecodeCfg &c,
                            size_t smem, cudaStream_t s, bool pdl, int grid);

// Registers per thread of each kernel instantiation (read once from the
// compiled kernel), for the residency estimate of the configuration search.
static int decode_regs(int dtype, bool asym, int R, int NB) {
    static std::mutex mu;
    static int cache[2][2][3][3];   // [dtype][asym][R - 1][log2 NB]
    const int ri = R - 1, ni = NB == 1 ? 0 : (NB == 2 ? 1 : 2);
    std::lock_guard<std::mutex> lk(mu);
    int &v = cache[dtype][asym ? 1 : 0][ri][ni];
    if (v == 0) {
        const void *f = nullptr;
#define W4A16_DK(D, A, RR, B) \
    if (dtype == D && asym == A && R == RR && NB == B) f = reinterpret_cast<const void *>(decode_kernel<D, A, RR, B>);
        W4A16_DK(0, false, 1, 1) W4A16_DK(0, false, 1, 2) W4A16_DK(0, false, 1, 4)
        W4A16_DK(0, false, 2, 1) W4A16_DK(0, false, 2, 2) W4A16_DK(0, false, 2, 4)
        W4A16_DK(0, true, 1, 1) W4A16_DK(0, true, 1, 2) W4A16_DK(0, true, 1, 4)
        W4A16_DK(0, true, 2, 1) W4A16_DK(0, true, 2, 2) W4A16_DK(0, true, 2, 4)
        W4A16_DK(1, false, 1, 1) W4A16_DK(1, false, 1, 2) W4A16_DK(1, false, 1, 4)
        W4A16_DK(1, false, 2, 1) W4A16_DK(1, false, 2, 2) W4A16_DK(1, false, 2, 4)
        W4A16_DK(1, true, 1, 1) W4A16_DK(1, true, 1, 2) W4A16_DK(1, true, 1, 4)
        W4A16_DK(1, true, 2, 1) W4A16_DK(1, true, 2, 2) W4A16_DK(1, true, 2, 4)
#undef W4A16_DK
        cudaFuncAttributes fa{};
        if (f == nullptr || cudaFuncGetAttributes(&fa, f) != cudaSuccess) {
            cudaGetLastError();
            return 128;                     // conservative; not cached
        }
        v = fa.numRegs > 0 ? fa.numRegs : 128;
    }
    return v;
}

// CTAs of configuration c that one SM holds at once: shared memory (plus the
// 1 KB the runtime reserves per CTA), threads, and registers (allocated per
// warp in units of 256).
static long long decode_per_sm(const DecodeCfg &c, int M, int K, int G, bool asym, int dtype, int smem_per_sm) {
    const long long smem = (long long)decode_smem_bytes(c, M, K, G, asym) + 1024;
    const int warps = c.NW + 1;
    const int regs = decode_regs(dtype, asym, c.R, c.NB);
    const long long warp_regs = ((regs * 32 + 255) / 256) * 256;
    long long n = smem_per_sm > 0 ? smem_per_sm / smem : 1;
    n = std::min(n, (long long)(64 / warps));
    n = std::min(n, 65536LL / (warps * warp_regs));
    return std::max(n, 0LL);
}

// Configuration from measured sweeps on GB300 (M = 1 decode, the Qwen3-4B-
// and Llama-3.1-8B-shaped layers, CUDA graphs with programmatic dependent
// launch, both per layer and over the four layers of a step in sequence,
// where a layer's CTAs must leave room for the next layer's to start early;
// the last search chose each layer's configuration by the time of the whole
// step, one layer at a time): one 16-row block per warp, 128-k boxes, K split
// into more cluster CTAs as N shrinks.  The whole grid should be resident on
// the SMs at once (a deeper ring that pushes CTAs into a second wave measured
// slower than a shallow one; at M >= 3 the staged activations of a long K
// row alone can do that): from the base choice, the ring is made as deep as
// it can be while the grid stays in one wave; failing that, fewer boxes per
// stage and then more cluster CTAs along K are tried, and the configuration
// with the fewest waves is kept.  Larger M (more staged activations and
// partials per CTA) measured faster with 128-row CTAs; MoE launches (slots > 1
// expert matrices of the same shape, one token each) have a base of their own.
DecodeCfg decode_pick_cfg(int M, int N, int K, int G, int sym, int dtype, int sm_count, int smem_per_sm,
                          int slots) {
    DecodeCfg b;
    if (slots > 1)                      // MoE: many small expert matrices, one token each
        b = K <= 1024 ? DecodeCfg{1, 2, 2, 4, 1} : DecodeCfg{1, 4, 4, 4, 2};
    else if (N >= 24576)
        b = M >= 3 ? DecodeCfg{1, 8, 1, 4, 2} : DecodeCfg{1, 4, 4, 2, 1};
    else if (N >= 16384)
        b = (M >= 2 && M <= 5) ? DecodeCfg{1, 8, 2, 3, 2} : DecodeCfg{1, 8, 4, 2, 2};
    else if (N >= 6144)
        b = M >= 2 ? DecodeCfg{1, 8, 4, 2, 5} : (K <= 3072 ? DecodeCfg{1, 8, 2, 4, 5} : DecodeCfg{1, 4, 4, 3, 4});
    else if (M >= 4 && M <= 6 && K >= 12288 && G <= 64) {
        // Long K with small groups: 128-row CTAs with K over a cluster of 8, or
        // of 4 when two such CTAs do not fit on an SM (the asymmetric G = 32
        // slice metadata is large).  Measured on 4096 x 14336 in CUDA graphs
        // with early launch: G = 64 symmetric 5-9 % faster than the rules
        // below at M = 4..6, G = 32 asymmetric 4-5 % at M = 4 and 16 % at
        // M = 5; at M = 3, 7 and 8, and at G = 128, the rules below stay best.
        b = DecodeCfg{1, 8, 2, 3, 8};
        const long long ctas8 = (long long)((N + 127) / 128) * 8;
        if (decode_per_sm(b, M, K, G, sym == 0, dtype, smem_per_sm) * sm_count < ctas8) b.S = 4;
    } else if (M >= 6 && K >= 8192)
        b = K >= 12288 ? DecodeCfg{1, 8, 4, 3, 4} : DecodeCfg{1, 8, 4, 4, 6};
    else if (M >= 3 && K >= 12288)
        b = DecodeCfg{1, 4, 4, 2, 6};
    else
        b = DecodeCfg{1, 4, 4, 4, 8};
    const bool asym = sym == 0;
    const int nblk = (K + kBoxK - 1) / kBoxK;
    while (b.S > 1 && nblk / b.S < 1) b.S >>= 1;            // at least one K block per CTA
    const int RT = 16 * b.R * b.NW;
    const long long tiles = (long long)((N + RT - 1) / RT) * std::max(slots, 1);
    DecodeCfg best = b;
    long long best_waves = -1;
    for (int S = b.S; S <= 8; S *= 2) {
        if (nblk / S < 1) break;
        const int nb = (nblk + S - 1) / S;
        for (int NB = b.NB; NB >= 1; NB >>= 1) {
            if (NB > nb && NB > 1) continue;                 // 4, 2 or 1 boxes per stage, <= the slice
            for (int NS = b.NS; NS >= 2; --NS) {
                DecodeCfg c{b.R, b.NW, NB, NS, S};
                if (!decode_cfg_valid(c, M, K, G, asym)) continue;
                const long long per_sm = decode_per_sm(c, M, K, G, asym, dtype, smem_per_sm);
                if (per_sm <= 0) continue;
                const long long waves = (tiles * S + per_sm * sm_count - 1) / (per_sm * sm_count);
                if (waves <= 1) return c;
                if (best_waves < 0 || waves < best_waves) {
                    best = c;
                    best_waves = waves;
                }
            }
        }
        if (S == 8) break;
    }
    if (best_waves < 0) {                                    // nothing valid: the smallest footprint
        best = DecodeCfg{b.R, b.NW, 1, 2, b.S};
        while (!decode_cfg_valid(best, M, K, G, asym) && best.S < 8) best.S *= 2;
    }
    return best;
}

template <int DT, bool ASYM, int R, int NB>
static cudaError_t launch_t(const DecodeMaps &tw, const DecodeParams &p, const DecodeCfg &c,
                            size_t smem, cudaStream_t s, bool pdl, int grid) {
    auto kern = decode_kernel<DT, ASYM, R, NB>;
    if (smem > 48 * 1024) {
        cudaError_t e = raise_smem_cap(reinterpret_cast<const void *>(kern), smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(32 * (c.NW + 1), 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, tw, p);
}

template <int DT, bool ASYM>
static cudaError_t launch_rnb(int R, int NB, const DecodeMaps &tw, const DecodeParams &p,
                              const DecodeCfg &c, size_t smem, cudaStream_t s, bool pdl, int grid) {
    if (R == 1) {
        switch (NB) {
            case 1: return launch_t<DT, ASYM, 1, 1>(tw, p, c, smem, s, pdl, grid);
            case 2: return launch_t<DT, ASYM, 1, 2>(tw, p, c, smem, s, pdl, grid);
            default: return launch_t<DT, ASYM, 1, 4>(tw, p, c, smem, s, pdl, grid);
        }
    }
    switch (NB) {
        case 1: return launch_t<DT, ASYM, 2, 1>(tw, p, c, smem, s, pdl, grid);
        case 2: return launch_t<DT, ASYM, 2, 2>(tw, p, c, smem, s, pdl, grid);
        default: return launch_t<DT, ASYM, 2, 4>(tw, p, c, smem, s, pdl, grid);
    }
}

static cudaError_t launch_dispatch(int dtype, bool asym, int R, int NB, const DecodeMaps &tw,
                                   const DecodeParams &p, const DecodeCfg &c, size_t smem,
                                   cudaStream_t s, bool pdl, int grid) {
    if (dtype == 0)
        return asym ? launch_rnb<0, true>(R, NB, tw, p, c, smem, s, pdl, grid)
                    : launch_rnb<0, false>(R, NB, tw, p, c, smem, s, pdl, grid);
    return asym ? launch_rnb<1, true>(R, NB, tw, p, c, smem, s, pdl, grid)
                : launch_rnb<1, false>(R, NB, tw, p, c, smem, s, pdl, grid);
}

#ifdef W4A16_DECODE_TRACE
// The timeline hook's buffer and traced (N, K) pairs (host side; set by
// decode_trace_install, read when a launch's parameters are built).
static unsigned long long *g_trace_buf = nullptr;
static int g_trace_nk[2 * kTraceLayers] = {};

static unsigned long long *decode_trace_slice(const GemmArgs &a) {
    if (g_trace_buf == nullptr || a.expert_ids != nullptr) return nullptr;
    for (int i = 0; i < kTraceLayers; ++i)
        if (g_trace_nk[2 * i] == a.N && g_trace_nk[2 * i + 1] == a.K)
            return g_trace_buf + (size_t)i * kTraceCtas * kTraceEvents;
    return nullptr;
}
#endif

cudaError_t launch_decode(const GemmArgs &a, const DecodeCfg &c, const DeviceInfo &dev,
                          cudaStream_t s, bool pdl, bool hold_copies) {
    if (dev.encode_tiled == nullptr) return cudaErrorNotSupported;
    const bool asym = a.qzeros != nullptr;
    const int RT = 16 * c.R * c.NW;
    DecodeMaps tw;
    const bool wide = a.K % kBoxK == 0;
    {
        EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(dev.encode_tiled);
        // rows as [N] or, with SiLU, as [2][I] (a dimension of 2 with stride I rows)
        const int silu = a.silu_mul ? 1 : 0;
        const cuuint64_t rows = silu ? (cuuint64_t)(a.N / 2)
                                     : (cuuint64_t)a.N * (a.expert_ids != nullptr ? (cuuint64_t)a.n_experts : 1);
        const cuuint64_t row_bytes = (cuuint64_t)(a.K / 8) * 4;
        const cuuint32_t box_rows = silu ? (cuuint32_t)(RT / 2) : (cuuint32_t)RT;
        cuuint64_t dims[3] = {(cuuint64_t)(a.K / 8), rows, 2};
        cuuint64_t strides[2] = {row_bytes, row_bytes * rows};
        cuuint32_t box[3] = {(cuuint32_t)(kBoxK / 8), box_rows, 2};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult r = encode(&tw.one, CU_TENSOR_MAP_DATA_TYPE_INT32, 2 + silu, const_cast<int32_t *>(a.qweight),
                            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        tw.wide = tw.one;
        if (wide) {
            // [blocks][(half)][row][16 words]
            cuuint64_t dw[4], sw[3];
            cuuint32_t bw[4];
            int nd = 0;
            dw[nd] = kBoxK / 8; bw[nd++] = kBoxK / 8;
            dw[nd] = rows; bw[nd] = box_rows; sw[nd - 1] = row_bytes; ++nd;
            if (silu) { dw[nd] = 2; bw[nd] = 2; sw[nd - 1] = row_bytes * rows; ++nd; }
            dw[nd] = (cuuint64_t)(a.K / kBoxK); bw[nd] = (cuuint32_t)c.NB; sw[nd - 1] = kBoxRowBytes; ++nd;
            r = encode(&tw.wide, CU_TENSOR_MAP_DATA_TYPE_INT32, nd, const_cast<int32_t *>(a.qweight), dw, sw, bw,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        }
    }
    DecodeParams p;
    p.x = (const uint16_t *)a.x;
    p.scales = (const uint16_t *)a.scales;
    p.qz = a.qzeros;
    p.out = (uint16_t *)a.out;
    p.bias = (const uint16_t *)a.bias;
    p.silu = a.silu_mul ? 1 : 0;
    p.hold = hold_copies ? 1 : 0;
#ifdef W4A16_DECODE_TRACE
    p.trace = decode_trace_slice(a);
#endif
    p.expert_ids = a.expert_ids;
    p.route_w = a.route_w;
    p.n_experts = a.n_experts;
    p.topk = a.topk;
    p.status = dev.status;
    p.dq = dq_consts_i4(a.dtype);
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = a.G;
    p.ng = a.K / a.G;
    p.log2G = a.G == 32 ? 5 : (a.G == 64 ? 6 : 7);
    p.NW = c.NW;
    p.NB = c.NB;
    p.NS = c.NS;
    p.S = c.S;
    p.nblk = (a.K + kBoxK - 1) / kBoxK;
    p.wide = wide ? 1 : 0;
    p.xpitch = decode_xpitch(c, a.K);
    p.gmax = decode_gmax(c, a.K, a.G);
    const int tiles = a.silu_mul ? (a.N / 2 + RT / 2 - 1) / (RT / 2) : (a.N + RT - 1) / RT;
    p.tiles = tiles;
    const long long grid_ll = (long long)tiles * c.S * (a.expert_ids != nullptr ? a.n_slots : 1);
    if (grid_ll > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    const int grid = (int)grid_ll;
    const size_t smem = decode_smem_bytes(c, a.M, a.K, a.G, asym);
    return launch_dispatch(a.dtype, asym, c.R, c.NB, tw, p, c, smem, s, pdl, grid);
}

cudaError_t decode_trace_install(unsigned long long *buf, const int *nk) {
#ifdef W4A16_DECODE_TRACE
    g_trace_buf = buf;
    for (int i = 0; i < 2 * kTraceLayers; ++i) g_trace_nk[i] = (buf != nullptr && nk != nullptr) ? nk[i] : 0;
    return cudaSuccess;
#else
    (void)nk;
    return buf == nullptr ? cudaSuccess : cudaErrorNotSupported;   // not compiled into this build
#endif
}

}  // namespace w4a16
