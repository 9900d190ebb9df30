// decode_stream.cu -- stream-K skinny-M (M <= 8) W4A16 GEMM for sm_103a.
//
// "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP skinny
// decode", PR description: batch sizes M <= 5 go to a skinny split-K GEMM
// optimised for single-token decode, reading the same packed [N, K/8]
// weights as the prefill path.  The skinny GEMM is bound by the weight
// stream ("a memory-bound kernel", "Upstream sync 67/N ... (conflict)",
// section "Upstream's Python side is kept -- and it does NOT work here").
//
// Design (GB300-first):
//  * Units of 32 weight rows x 256 k (4 KB packed) are ordered row block by
//    row block.  One CTA runs per SM; CTA c takes the contiguous unit range
//    [c U / C, (c+1) U / C) and its eight warps split that range into
//    contiguous pieces, so every SM and every warp streams the same number
//    of bytes to within one unit.
//  * Every warp streams its own units: it owns D shared-memory slots, keeps
//    them filled with one 3-D TMA copy per unit (two 128-k boxes of 32 rows,
//    64 bytes a row), copies a unit into registers as soon as it lands and
//    refills the slot at once, so D units per warp (8 D per SM) are in flight
//    nearly all the time.  (A TMA copy instruction holds its issuing warp for
//    a few hundred cycles whatever its size, so eight issuing warps, not one,
//    are what keeps the HBM stream busy.)  Scales and zero points are read
//    with plain loads one unit ahead.
//  * The warps dequantise in registers (dq_word_i4_rt: RN((q - z) s) per
//    weight, bit for bit the definition) and multiply on the tensor cores
//    with mma.sync m16n8k16 (fp32 accumulate), two 16-row blocks per warp and
//    two accumulator chains each.  x (all of K, permuted to the dequantiser's
//    (k, k+4) nibble pairing) is staged once per CTA.
//  * Reduction, deterministic and without waiting: a row block one warp
//    covers is stored directly; one split between warps of the CTA is summed
//    from their shared-memory slots in warp order; one split between CTAs
//    (at most the first and the last of each CTA) leaves the CTA's partial in
//    a global workspace, and the CTA that arrives last on the block's ticket
//    sums every CTA's partial in CTA order, stores y and resets the ticket.
//  * Programmatic dependent launch: weights, scales and zero points stream
//    before the grid-dependency wait; x, y and the workspace are touched only
//    after it.  Weights, scales and zero points must therefore not be written
//    by the kernel that immediately precedes this one on the stream.
//  * Every mbarrier wait is bounded; a wait that runs out sets the device
//    status word and the CTA's abort flag, and every warp leaves its loop
//    (after its copies in flight have landed).
#include <cuda.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "skinny.cuh"

namespace w4a16 {
namespace stream {

constexpr int kRows = 32;                          // weight rows per unit
constexpr int kUnitK = 256;                        // k per unit
constexpr int kBoxBytes = kRows * 64;              // one 128-k box: 32 rows x 64 B
constexpr int kUnitBytes = 2 * kBoxBytes;          // 4 KB
constexpr int kNW = 8;                             // warps per CTA
constexpr int kThreads = 32 * kNW;
constexpr int kSlot = kRows * 8;                   // floats per partial slot: [32 rows][8 m]
constexpr int kMaxD = 4;

constexpr int kMaxCTAs = 256;                      // grid size limit (CTA range table)
constexpr int kMetaSlots = 3;                      // per-warp metadata ring: units ahead

struct Params {
    const uint16_t *x;
    const uint16_t *scales;
    const int32_t *qz;
    uint16_t *out;
    float *ws;            // CTA partial slots [C][2][32][8]
    int *cnt;             // tickets [ceil(N / 32)], zero between calls
    int *status;
    DqConsts dq;
    int U;                // total units
    int C;                // CTAs
    int M, N, K, G, ng, log2G;
    int ukc;              // units per row block (K / 256)
    int xpitch;           // bytes per staged x row
    int mstride;          // bytes of one unit's metadata
    int cstart[kMaxCTAs + 1];   // CTA c takes units [cstart[c], cstart[c + 1])
};

// Metadata of one unit in shared memory: scales [32 rows][256 / G] (dtype
// bits), then for asymmetric weights zero-point words [4 row octets][256 / G].
__host__ __device__ inline int meta_scale_bytes(int G) { return kRows * (512 / G); }
__host__ __device__ inline int meta_bytes(int G, bool asym) {
    return meta_scale_bytes(G) + (asym ? 4 * (1024 / G) : 0);
}

struct Layout {
    uint32_t ring, meta, x, slots, bars, total;
};

__host__ __device__ inline Layout stream_layout(int D, int M, int xpitch, int mstride) {
    Layout L;
    uint32_t off = 0;
    L.ring = off;                                   // 128-B aligned (TMA destination)
    off += (uint32_t)kNW * D * kUnitBytes;
    L.meta = off;                                   // [kNW][kMetaSlots][mstride]
    off += (uint32_t)kNW * kMetaSlots * mstride;
    off = (off + 15u) & ~15u;
    L.x = off;                                      // [M][xpitch]
    off += (uint32_t)M * xpitch;
    off = (off + 15u) & ~15u;
    L.slots = off;                                  // [kNW][2][32][M] fp32 warp partials
    off += (uint32_t)kNW * 2 * kRows * M * 4;
    off = (off + 15u) & ~15u;
    L.bars = off;                                   // full[kNW D], abort flag, range tables
    off += (uint32_t)kNW * D * 8 + 16 + 4 * (2 * kNW + 1);
    L.total = off + 128;                            // slack to align the base to 128
    return L;
}

// The CTA whose range contains unit u (binary search of the range table).
__device__ __forceinline__ int cta_of(int u, const Params &p) {
    int lo = 0, hi = p.C - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cstart[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// cp.async of 4, 8 or 16 bytes; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async(uint32_t dst, const void *src, int bytes, int src_bytes) {
    if (bytes == 16)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
    else if (bytes == 8)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Wait for a phase for at most kDrainLimitNs, ignoring the CTA's abort flag:
// used only to let issued copies land before the CTA exits.
constexpr unsigned long long kDrainLimitNs = 100000000ull;  // 100 ms
__device__ __forceinline__ void mbar_drain_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 255u) == 0 && globaltimer() - t0 > kDrainLimitNs) return;
    }
}

// This lane's share of the metadata of the unit at (rb, kc): row `lane`'s
// scales of the unit (4, 8 or 16 bytes, one copy) and, for asymmetric
// weights, lanes 0..3 (0..7 for G = 32) one octet's zero-point words.  Rows
// past N read as zeros.
template <bool ASYM>
__device__ __forceinline__ void copy_meta(uint32_t dst, const Params &p, int rb, int kc, int lane) {
    const int gsh = 8 - p.log2G;                    // log2(groups per unit)
    const int sbytes = 2 << gsh;
    const int row = rb * kRows + lane;
    const bool v = row < p.N;
    cp_async(dst + (uint32_t)lane * sbytes, p.scales + (v ? (size_t)row * p.ng + ((size_t)kc << gsh) : 0), sbytes,
             v ? sbytes : 0);
    if (ASYM) {
        const int zbytes = 4 << gsh;                // one octet's words: 8, 16 or 32 B
        const int nz = zbytes > 16 ? 8 : 4;
        if (lane < nz) {
            const int oc = lane & 3, part = lane >> 2;
            const int octet = rb * 4 + oc;
            const bool vz = octet * 8 < p.N;
            const int cb = zbytes > 16 ? 16 : zbytes;
            cp_async(dst + (uint32_t)(kRows * sbytes + oc * zbytes + part * 16),
                     p.qz + (vz ? (size_t)octet * p.ng + ((size_t)kc << gsh) + part * 4 : 0), cb, vz ? cb : 0);
        }
    }
}

template <int DT, bool ASYM, int D>
__global__ void __launch_bounds__(kThreads, 2) decode_stream_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                  const __grid_constant__ Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int ukc = p.ukc, M = p.M;
    const Layout L = stream_layout(D, M, p.xpitch, p.mstride);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L.bars;
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bars + 8 * kNW * D);
    // wtab[w] = first unit of warp w (wtab[kNW] = end of the CTA's range);
    // wrb[w] = its row block.
    int *wtab = reinterpret_cast<int *>(smem + L.bars + 8 * kNW * D + 16);
    int *wrb = wtab + kNW + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNW * D; ++s) mbar_init(full(s), 1);   // the issuing lane's arrive + tx bytes
        *abort_flag = 0;
        const int cu0 = p.cstart[blockIdx.x];
        const int n_cta = p.cstart[blockIdx.x + 1] - cu0;
        for (int w = 0; w <= kNW; ++w) wtab[w] = cu0 + (n_cta * w) / kNW;
        for (int w = 0; w < kNW; ++w) wrb[w] = wtab[w] / ukc;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependents_launch();

    const int n_units = wtab[warp + 1] - wtab[warp];
    const int rb0 = wrb[warp], kc0 = wtab[warp] - rb0 * ukc;
    auto advance = [&](int &rbv, int &kcv) {
        if (++kcv == ukc) { kcv = 0; ++rbv; }
    };
    // Weight copies: the unit at (irb, ikc) into ring slot `slot` (lane 0).
    // The arrive is relaxed: it orders nothing but the copy.
    int irb = rb0, ikc = kc0;                       // position of the next unit to copy
    auto issue_next = [&](int slot) {
        asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(full(slot)),
                     "r"((uint32_t)kUnitBytes)
                     : "memory");
        tma_load_3d(sbase + L.ring + (uint32_t)slot * kUnitBytes, &wmap, full(slot), 0, irb * kRows, ikc * 2);
    };
    int issued = D < n_units ? D : n_units;        // units whose weight copies have been issued
    if (lane == 0 && warp == 0) tma_prefetch_desc(&wmap);
    for (int j = 0; j < issued; ++j) {
        if (lane == 0) issue_next(warp * D + j);
        advance(irb, ikc);
    }
    // Metadata copies: kMetaSlots units ahead, one commit group per unit
    // (empty groups past the end keep the group count regular).
    const uint32_t meta_w = sbase + L.meta + (uint32_t)(warp * kMetaSlots) * p.mstride;
    int mrb = rb0, mkc = kc0;                       // position of the next unit's metadata
#pragma unroll
    for (int j = 0; j < kMetaSlots; ++j) {
        if (j < n_units) copy_meta<ASYM>(meta_w + (uint32_t)j * p.mstride, p, mrb, mkc, lane);
        cp_async_commit();
        advance(mrb, mkc);
    }

    // ---- x -> shared memory, permuted to the (k, k+4) pairing
    grid_dependency_wait();
    {
        unsigned char *xs = smem + L.x;
        const int nch = p.K / 8;                   // 16-byte chunks per row
        for (int m = 0; m < M; ++m)
            for (int c = threadIdx.x; c < nch; c += kThreads) {
                const uint4 v = *reinterpret_cast<const uint4 *>(p.x + (size_t)m * p.K + 8 * c);
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
    __syncthreads();

    // Lanes whose batch column g is >= M read x row 0: their MMA output
    // columns are never stored.
    const unsigned char *xrow = smem + L.x + (size_t)(g < M ? g : 0) * p.xpitch + t * 16;
    const uint32_t zl_sym = zlo2<DT>(8u), zh_sym = zhi2<DT>(8u);
    const DqConsts dc = p.dq;
    float *slots = reinterpret_cast<float *>(smem + L.slots);       // [kNW][2][32][M]
    float *wslots = slots + (size_t)warp * 2 * kRows * M;
    const int gsh = 8 - p.log2G;
    const int sbytes = 2 << gsh;
    const int go0 = (32 * t) >> p.log2G, go1 = (128 + 32 * t) >> p.log2G;   // the lane's groups in the unit

    int rb = rb0, kc = kc0;                          // position of the unit being consumed
    int kc_first = kc;
    float acc[2][2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[a][c][e] = 0.f;

    // Emit row block frb (units kc_first .. kc_last of it): directly if this
    // warp covered it completely, else into this warp's partial slot.
    auto flush = [&](int frb, int kc_last) {
        float c[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) c[h][e] = chain_sum<2>(acc[h], e);
        const bool whole = kc_first == 0 && kc_last == ukc - 1;
        float *slot = wslots + (frb == rb0 ? 0 : kRows * M);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = h * 16 + g + (e >= 2 ? 8 : 0), m = 2 * t + (e & 1);
                if (m < M) {
                    if (!whole) slot[r * M + m] = c[h][e];
                    else if (frb * kRows + r < p.N) p.out[(size_t)m * p.N + frb * kRows + r] = f32_to_dt<DT>(c[h][e]);
                }
            }
    };

    bool ok = true;
    int s = 0;                                       // ring slot of the unit being consumed
    uint32_t par = 0u;                               // its phase parity
    int ms = 0;                                      // metadata slot of the unit being consumed
    for (int j = 0; j < n_units; ++j) {
        if (kc == 0 && j > 0) {              // a new row block begins
            flush(rb - 1, ukc - 1);
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[a][c][e] = 0.f;
            kc_first = 0;
        }
        // ---- this unit's scales and zero points: copied kMetaSlots units ago
        cp_async_wait<kMetaSlots - 1>();
        __syncwarp();
        const unsigned char *meta = smem + L.meta + (size_t)(warp * kMetaSlots + ms) * p.mstride;
        uint32_t sc[4][2];                           // [row g + 8 i][128-k half]
        uint32_t zw[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const unsigned char *sr = meta + (i * 8 + g) * sbytes;
            sc[i][0] = *reinterpret_cast<const uint16_t *>(sr + go0 * 2);
            sc[i][1] = *reinterpret_cast<const uint16_t *>(sr + go1 * 2);
            if (ASYM) {
                const unsigned char *zr = meta + kRows * sbytes + i * (4 << gsh);
                zw[i][0] = *reinterpret_cast<const uint32_t *>(zr + go0 * 4);
                zw[i][1] = *reinterpret_cast<const uint32_t *>(zr + go1 * 4);
            }
        }
        // the slot's values are in registers: refill it with the unit
        // kMetaSlots ahead
        asm volatile("" ::"r"(sc[0][0]), "r"(sc[1][1]), "r"(sc[2][0]), "r"(sc[3][1]) : "memory");
        __syncwarp();
        if (j + kMetaSlots < n_units) copy_meta<ASYM>(meta_w + (uint32_t)ms * p.mstride, p, mrb, mkc, lane);
        cp_async_commit();
        advance(mrb, mkc);
        if (++ms == kMetaSlots) ms = 0;

        // ---- the unit's weights
        const int slot = warp * D + s;
        if (!mbar_wait_bounded(full(slot), par, p.status, abort_flag)) {
            ok = false;
            break;
        }
        // The whole unit into registers, then the slot is refilled at once.
        const unsigned char *stage = smem + L.ring + (size_t)slot * kUnitBytes + g * 64 + t * 16;
        uint4 wv[2][2][2];                          // [128-k half][16-row block][row g / g + 8]
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                wv[kb][h][0] = sh_v4(stage + kb * kBoxBytes + h * 16 * 64);
                wv[kb][h][1] = sh_v4(stage + kb * kBoxBytes + (h * 16 + 8) * 64);
            }
        if (issued < n_units) {
            // This warp's loads from the slot have returned (the asm consumes
            // them) and are ordered before the async-proxy copy that refills it.
            asm volatile("" ::"r"(wv[0][0][0].x), "r"(wv[0][0][1].x), "r"(wv[0][1][0].x), "r"(wv[0][1][1].x),
                         "r"(wv[1][0][0].x), "r"(wv[1][0][1].x), "r"(wv[1][1][0].x), "r"(wv[1][1][1].x)
                         : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) issue_next(slot);
            advance(irb, ikc);
            ++issued;
        }
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            const unsigned char *xb = xrow + (size_t)(kc * 2 + kb) * 256;
            const uint4 xv[4] = {sh_v4(xb), sh_v4(xb + 64), sh_v4(xb + 128), sh_v4(xb + 192)};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t zla = zl_sym, zha = zh_sym, zlb = zl_sym, zhb = zh_sym;
                if (ASYM) {
                    const uint32_t za = (zw[2 * h][kb] >> (4 * g)) & 0xFu;
                    const uint32_t zb = (zw[2 * h + 1][kb] >> (4 * g)) & 0xFu;
                    zla = zlo2<DT>(za); zha = zhi2<DT>(za);
                    zlb = zlo2<DT>(zb); zhb = zhi2<DT>(zb);
                }
                mac_block<DT, 2>(acc[h], dc, wv[kb][h][0], wv[kb][h][1], zla, zha, rep2(sc[2 * h][kb]), zlb, zhb,
                                 rep2(sc[2 * h + 1][kb]), xv);
            }
        }
        advance(rb, kc);
        if (++s == D) { s = 0; par ^= 1u; }
    }
    cp_async_wait<0>();                              // no metadata copy outlives the CTA
    if (n_units > 0 && ok) {
        const int last_rb = (kc == 0) ? rb - 1 : rb;
        const int last_kc = (kc == 0) ? ukc - 1 : kc - 1;
        flush(last_rb, last_kc);
    }
    __syncthreads();
    if (*abort_flag) {
        // Copies this warp issued may still be in flight: wait (bounded) for
        // the last phase armed on each of its slots before the CTA leaves.
        if (lane == 0)
            for (int r = 0; r < D && r < issued; ++r) {
                const int last_j = ((issued - 1 - r) / D) * D + r;   // last unit that used slot r
                mbar_drain_bounded(full(warp * D + r), (uint32_t)((last_j / D) & 1));
            }
        return;
    }

    // ---- row blocks split between warps: sum the warps' slots in warp order.
    // Row blocks of this CTA: rb_lo .. rb_hi; warp (rbl % kNW) handles rb_lo + rbl.
    const int cu0 = wtab[0], cu1 = wtab[kNW];
    if (cu1 == cu0) return;
    const int rb_lo = cu0 / ukc, rb_hi = (cu1 - 1) / ukc;
    const int nel = kRows * M;                      // elements of a row block's partial: [32][M]
    for (int rbl = warp; rbl <= rb_hi - rb_lo; rbl += kNW) {
        const int frb = rb_lo + rbl;
        const int ub0 = frb * ukc, ub1 = ub0 + ukc;   // the block's units
        unsigned pieces = 0;                          // warps holding a partial piece of it
        for (int w = 0; w < kNW; ++w) {
            const int a = wtab[w], b = wtab[w + 1];
            if (a < b && a < ub1 && b > ub0 && !(a <= ub0 && b >= ub1)) pieces |= 1u << w;
        }
        if (pieces == 0) continue;                    // stored directly by its warp
        const bool cta_complete = cu0 <= ub0 && cu1 >= ub1;
        const int side = (frb == rb_lo) ? 0 : 1;
        float *gslot = p.ws + ((size_t)blockIdx.x * 2 + side) * kSlot;
        for (int e = lane; e < nel; e += 32) {
            const int r = e / M, m = e - r * M;
            float sum = 0.f;
            for (int w = 0; w < kNW; ++w)
                if (pieces & (1u << w)) sum += slots[((size_t)w * 2 + (frb == wrb[w] ? 0 : 1)) * nel + e];
            const int row = frb * kRows + r;
            if (cta_complete) {
                if (row < p.N) p.out[(size_t)m * p.N + row] = f32_to_dt<DT>(sum);
            } else {
                gslot[r * 8 + m] = sum;
            }
        }
        if (cta_complete) continue;
        // ---- split between CTAs: ticket; the last CTA sums every CTA's
        // partial in CTA order.  The warp barrier orders every lane's partial
        // before lane 0's release-acquire increment; the acquire and the
        // barrier after it order the last CTA's loads after the others'
        // partials.
        const int cf = cta_of(ub0, p), cl = cta_of(ub1 - 1, p);
        __syncwarp();
        int ticket = 0;
        if (lane == 0)
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(ticket) : "l"(p.cnt + frb) : "memory");
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket != cl - cf) continue;
        __syncwarp();
        float sums[kRows * 8 / 32];                   // this lane's elements e = lane + 32 i
#pragma unroll
        for (int i = 0; i < kRows * 8 / 32; ++i) sums[i] = 0.f;
        for (int c = cf; c <= cl; ++c) {
            const int crb_lo = p.cstart[c] / ukc;
            const float *cs = p.ws + ((size_t)c * 2 + (frb == crb_lo ? 0 : 1)) * kSlot;
#pragma unroll
            for (int i = 0; i < kRows * 8 / 32; ++i) {
                const int e = lane + 32 * i;
                if (e < nel) {
                    const int r = e / M, m = e - r * M;
                    sums[i] += __ldcg(cs + r * 8 + m);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRows * 8 / 32; ++i) {
            const int e = lane + 32 * i;
            if (e < nel) {
                const int r = e / M, m = e - r * M;
                const int row = frb * kRows + r;
                if (row < p.N) p.out[(size_t)m * p.N + row] = f32_to_dt<DT>(sums[i]);
            }
        }
        if (lane == 0) p.cnt[frb] = 0;
    }
}

}  // namespace stream

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Shared memory a CTA may use so that two of them (this layer's and the next
// one's, under programmatic dependent launch) fit on one SM together.
constexpr size_t kStreamSmemBudget = 110 * 1024;

static int stream_xpitch(int K) { return ((K * 2 + 127) / 128) * 128 + 64; }   // odd multiple of 64

size_t decode_stream_smem_bytes(int M, int K, int G, bool asym, int D) {
    return stream::stream_layout(D, M, stream_xpitch(K), stream::meta_bytes(G, asym)).total;
}

int decode_stream_pick_d(int M, int K, int G, bool asym) {
    for (int D = stream::kMaxD; D >= 2; --D)
        if (decode_stream_smem_bytes(M, K, G, asym, D) <= kStreamSmemBudget) return D;
    return 0;
}

bool decode_stream_applicable(int M, int N, int K, int G, bool asym) {
    if (M < 1 || M > 8 || K % stream::kUnitK != 0) return false;
    if ((N + stream::kRows - 1) / stream::kRows > kDecodeTickets) return false;
    if ((long long)((N + stream::kRows - 1) / stream::kRows) * (K / stream::kUnitK) >= (1LL << 31)) return false;
    return decode_stream_pick_d(M, K, G, asym) >= 2;
}

size_t decode_stream_workspace_floats(int sm_count) { return (size_t)sm_count * 2 * stream::kSlot; }

template <int DT, bool ASYM, int D>
static cudaError_t launch_stream_t(const CUtensorMap &map, const stream::Params &p, size_t smem, cudaStream_t s,
                                   bool pdl) {
    auto kern = stream::decode_stream_kernel<DT, ASYM, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.C, 1, 1);
    cfg.blockDim = dim3(stream::kThreads, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, map, p);
}

template <int DT, bool ASYM>
static cudaError_t launch_stream_d(int D, const CUtensorMap &map, const stream::Params &p, size_t smem,
                                   cudaStream_t s, bool pdl) {
    if (D == 2) return launch_stream_t<DT, ASYM, 2>(map, p, smem, s, pdl);
    if (D == 3) return launch_stream_t<DT, ASYM, 3>(map, p, smem, s, pdl);
    return launch_stream_t<DT, ASYM, 4>(map, p, smem, s, pdl);
}

cudaError_t launch_decode_stream(const GemmArgs &a, int D, const DeviceInfo &dev, float *ws, int *cnt,
                                 cudaStream_t s, bool pdl) {
    if (dev.encode_tiled == nullptr) return cudaErrorNotSupported;
    const bool asym = a.qzeros != nullptr;
    if (!decode_stream_applicable(a.M, a.N, a.K, a.G, asym)) return cudaErrorInvalidValue;
    if (D <= 0) D = decode_stream_pick_d(a.M, a.K, a.G, asym);
    if (D < 2 || D > stream::kMaxD) return cudaErrorInvalidValue;
    if (decode_stream_smem_bytes(a.M, a.K, a.G, asym, D) > (size_t)dev.max_smem_optin) return cudaErrorInvalidValue;
    CUtensorMap map;
    {
        // qweight viewed as [K / 128 blocks][N rows][16 words]; a box is two
        // consecutive blocks of 32 rows (rows past N read as zeros).
        EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(dev.encode_tiled);
        cuuint64_t dims[3] = {16, (cuuint64_t)a.N, (cuuint64_t)(a.K / 128)};
        cuuint64_t strides[2] = {(cuuint64_t)(a.K / 8) * 4, 64};
        cuuint32_t box[3] = {16, (cuuint32_t)stream::kRows, 2};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, const_cast<int32_t *>(a.qweight), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    stream::Params p;
    p.x = (const uint16_t *)a.x;
    p.scales = (const uint16_t *)a.scales;
    p.qz = a.qzeros;
    p.out = (uint16_t *)a.out;
    p.ws = ws;
    p.cnt = cnt;
    p.status = dev.status;
    p.dq = dq_consts_i4(a.dtype);
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = a.G;
    p.ng = a.K / a.G;
    p.log2G = a.G == 32 ? 5 : (a.G == 64 ? 6 : 7);
    p.ukc = a.K / stream::kUnitK;
    p.xpitch = stream_xpitch(a.K);
    p.mstride = stream::meta_bytes(a.G, asym);
    const int rblocks = (a.N + stream::kRows - 1) / stream::kRows;
    p.U = rblocks * p.ukc;
    int grid = dev.sm_count < stream::kMaxCTAs ? dev.sm_count : stream::kMaxCTAs;
    if (grid > p.U) grid = p.U;
    p.C = grid;
    for (int c = 0; c <= grid; ++c) p.cstart[c] = (int)((long long)c * p.U / grid);
    const size_t smem = decode_stream_smem_bytes(a.M, a.K, a.G, asym, D);
    if (a.dtype == 0)
        return asym ? launch_stream_d<0, true>(D, map, p, smem, s, pdl) : launch_stream_d<0, false>(D, map, p, smem, s, pdl);
    return asym ? launch_stream_d<1, true>(D, map, p, smem, s, pdl) : launch_stream_d<1, false>(D, map, p, smem, s, pdl);
}

}  // namespace w4a16
