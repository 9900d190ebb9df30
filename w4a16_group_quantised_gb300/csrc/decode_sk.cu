// decode_sk.cu -- balanced skinny-M W4A16 GEMM for sm_103a (M <= 8).
//
// Same operation and arithmetic as decode.cu ("[ROCm][Kernel] Add
// HybridW4A16LinearKernel: Triton prefill + HIP skinny decode", PR
// description: the skinny split-K GEMM for single-token decode), with the
// work divided so that every SM streams the same number of weight bytes:
//
//  * The weight matrix is cut into units of 16 rows x 128 k (1 KB packed),
//    ordered row block by row block.  One CTA of NW warps runs per SM; CTA c
//    takes the contiguous unit range [c U / C, (c+1) U / C), equal shares to
//    +-1 unit, so no SM waits for another at the end.  Inside the CTA the
//    warps split the range into contiguous pieces.
//  * Each lane streams its share of a unit (16 bytes of rows g and g+8, plus
//    their scales and zero points) with non-allocating 128-bit loads through
//    an NS-deep register ring, so every warp keeps NS units in flight from
//    its first cycle.  (Plain loads, not TMA: a TMA box costs a fixed few
//    hundred nanoseconds of the SM's copy engine, so 1 KB boxes cannot feed
//    the HBM rate.)  x (all of K, permuted to the dequantiser's nibble
//    pairing) is staged once per CTA.
//  * Dequantisation (dq_word_i4) and the tensor-core MAC (mma.sync
//    m16n8k16, fp32 accumulate) are those of decode.cu.
//  * A row block that one warp covers completely is written out directly.
//    A row block split between warps of the CTA is summed from their partial
//    slots in shared memory, in warp order.  A row block split between CTAs
//    (at most the first and the last of each CTA) leaves the CTA's partial
//    in a global workspace; the CTA that arrives last on the block's counter
//    (an atomic ticket) sums every CTA's partial in CTA order, writes the
//    outputs and resets the counter to zero for the next call.  The order of
//    every sum is fixed, so results are deterministic, and no CTA ever waits
//    for another.
//  * Programmatic dependent launch: the first NS units of weights, scales and
//    zero points are requested before the grid-dependency wait; x, out and
//    the workspace are touched only after it.
#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace w4a16 {
namespace sk {

constexpr int kUnitK = 128;                          // k per unit
constexpr int kUnitRows = 16;
constexpr int kNW = 16;                              // warps per CTA
constexpr int kSlot = 128;                           // floats per partial slot: [16 rows][8 m]

struct Params {
    const uint16_t *x;
    const uint16_t *scales;
    const int32_t *qz;
    uint16_t *out;
    float *ws;            // CTA partial slots [C][2][16][8]
    int *counters;        // [N / 16], zero between calls
    int *status;
    long long U;          // total units
    int C;                // CTAs
    int M, N, K, G, ng, log2G;
    int nblk;             // units per row block (K blocks of 128; the last may be partial)
    int xpitch;           // bytes per x row in shared memory
};

template <int DT>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    if (DT == 0) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

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

template <int DT>
__device__ __forceinline__ uint32_t zhi_from_zlo(uint32_t zl2) {
    return ((zl2 & 0x000F000Fu) << (DT == 0 ? 4 : 3)) | rep2(Dtype<DT>::kMagicHi);
}

__host__ __device__ inline long long range_start(long long i, long long n, long long parts) {
    return i * n / parts;
}

// The CTA whose range contains unit u.
__device__ inline int cta_of(long long u, long long U, int C) {
    long long c = u * C / U;
    while (c + 1 < C && range_start(c + 1, U, C) <= u) ++c;
    while (c > 0 && range_start(c, U, C) > u) --c;
    return (int)c;
}

struct Layout {
    uint32_t x, slots, total;
};

__host__ __device__ inline Layout sk_layout(int M, int xpitch) {
    Layout L;
    uint32_t off = 0;
    L.x = off;                                               // [M][xpitch]
    off += (uint32_t)M * xpitch;
    off = (off + 15u) & ~15u;
    L.slots = off;                                           // [NW][2][16][8] fp32
    off += (uint32_t)kNW * 2 * kSlot * 4;
    L.total = off + 128;
    return L;
}

// One unit of a lane: 4 packed words of rows g and g+8 (32 k each), and the
// scale bits / zero-point words of those rows for the lane's group.
struct Slot {
    uint4 wa, wb;
    uint32_t sa, sb, za, zb;
};

template <bool ASYM>
__device__ __forceinline__ void load_unit(Slot &sl, const int32_t *qw, const Params &p, int urb, int ukb,
                                          int g, int t) {
    const int ra = urb * kUnitRows + g, rbw = ra + 8;
    const int k = ukb * kUnitK + 32 * t;
    const bool kin = k < p.K;
    const bool va = kin && ra < p.N, vb = kin && rbw < p.N;
    const size_t K8 = (size_t)(p.K >> 3);
    const int word = k >> 3;
    const int grp = k >> p.log2G;
    sl.wa = va ? ldg_stream_v4(qw + (size_t)ra * K8 + word) : make_uint4(0, 0, 0, 0);
    sl.wb = vb ? ldg_stream_v4(qw + (size_t)rbw * K8 + word) : make_uint4(0, 0, 0, 0);
    sl.sa = va ? (uint32_t)__ldg(p.scales + (size_t)ra * p.ng + grp) : 0u;
    sl.sb = vb ? (uint32_t)__ldg(p.scales + (size_t)rbw * p.ng + grp) : 0u;
    if (ASYM) {
        sl.za = va ? (uint32_t)__ldg(p.qz + (size_t)(ra >> 3) * p.ng + grp) : 0u;
        sl.zb = vb ? (uint32_t)__ldg(p.qz + (size_t)(rbw >> 3) * p.ng + grp) : 0u;
    }
}

template <int DT, bool ASYM, int NS>
__global__ void __launch_bounds__(kNW * 32, 1) decode_sk_kernel(const int32_t *__restrict__ qw,
                                                                const Params p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const Layout L = sk_layout(p.M, p.xpitch);
    const int nblk = p.nblk;

    const long long cu0 = range_start(blockIdx.x, p.U, p.C);
    const long long cu1 = range_start(blockIdx.x + 1, p.U, p.C);
    const int n_cta = (int)(cu1 - cu0);
    const int wu0 = (int)range_start(warp, n_cta, kNW);         // CTA-local units of this warp
    const int wu1 = (int)range_start(warp + 1, n_cta, kNW);
    const int n_units = wu1 - wu0;

    grid_dependents_launch();

    // unit -> (row block, k block) of this warp's first unit, then advanced incrementally
    const long long ufirst = cu0 + wu0;
    int rb = (int)(ufirst / nblk), kb = (int)(ufirst - (ufirst / nblk) * nblk);

    // ---- first NS units of weights, scales and zero points (static: before the dependency wait)
    Slot ring[NS];
    int rb_ahead = rb, kb_ahead = kb;   // the unit NS ahead, for refills
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        if (s < n_units) load_unit<ASYM>(ring[s], qw, p, rb_ahead, kb_ahead, g, t);
        if (++kb_ahead == nblk) { kb_ahead = 0; ++rb_ahead; }
    }

    // ---- x -> shared memory, permuted to the (k, k+4) pairing; zero beyond K
    grid_dependency_wait();
    {
        unsigned char *xs = smem + L.x;
        const int nch = nblk * 16;                 // 16-byte chunks per row
        for (int i = threadIdx.x; i < p.M * nch; i += blockDim.x) {
            const int m = i / nch, c = i - (i / nch) * nch;
            const int k = 8 * c;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (k < p.K) v = *reinterpret_cast<const uint4 *>(p.x + (size_t)m * p.K + k);
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

    const bool has_x = g < p.M;
    const unsigned char *xrow = smem + L.x + (size_t)g * p.xpitch + t * 16;
    const uint32_t zl_sym = zlo2<DT>(8u), zh_sym = zhi2<DT>(8u);
    const int first_rb = rb;
    float *wslots = reinterpret_cast<float *>(smem + L.slots) + (size_t)warp * 2 * kSlot;

    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    int kb_first = kb;

    // Emit the row block accumulated so far (kb_first .. kb_last): directly if
    // this warp covered it completely, else into this warp's partial slot.
    auto flush = [&](int frb, int kb_last) {
        float c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e] = acc[e] + acc2[e];
        if (kb_first == 0 && kb_last == nblk - 1) {
            const int row_a = frb * kUnitRows + g, row_b = row_a + 8, m0 = 2 * t;
            if (m0 < p.M) {
                if (row_a < p.N) p.out[(size_t)m0 * p.N + row_a] = f32_to_dt<DT>(c[0]);
                if (row_b < p.N) p.out[(size_t)m0 * p.N + row_b] = f32_to_dt<DT>(c[2]);
            }
            if (m0 + 1 < p.M) {
                if (row_a < p.N) p.out[(size_t)(m0 + 1) * p.N + row_a] = f32_to_dt<DT>(c[1]);
                if (row_b < p.N) p.out[(size_t)(m0 + 1) * p.N + row_b] = f32_to_dt<DT>(c[3]);
            }
            return;
        }
        float *slot = wslots + (frb == first_rb ? 0 : kSlot);
        slot[g * 8 + 2 * t] = c[0];
        slot[g * 8 + 2 * t + 1] = c[1];
        slot[(g + 8) * 8 + 2 * t] = c[2];
        slot[(g + 8) * 8 + 2 * t + 1] = c[3];
    };

    for (int i0 = 0; i0 < n_units; i0 += NS) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const int i = i0 + s;
            if (i < n_units) {
                if (kb == 0 && i > 0) {          // a new row block begins
                    flush(rb - 1, nblk - 1);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[e] = acc2[e] = 0.f;
                    kb_first = 0;
                }
                const Slot cur = ring[s];
                if (i + NS < n_units) load_unit<ASYM>(ring[s], qw, p, rb_ahead, kb_ahead, g, t);
                if (++kb_ahead == nblk) { kb_ahead = 0; ++rb_ahead; }

                uint32_t zla = zl_sym, zha = zh_sym, zlb = zl_sym, zhb = zh_sym;
                if (ASYM) {
                    const uint32_t za = (cur.za >> (4 * g)) & 0xFu, zb = (cur.zb >> (4 * g)) & 0xFu;
                    zla = zlo2<DT>(za); zha = zhi2<DT>(za);
                    zlb = zlo2<DT>(zb); zhb = zhi2<DT>(zb);
                }
                const uint32_t s2a = rep2(cur.sa), s2b = rep2(cur.sb);
                uint4 xv[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    xv[w] = make_uint4(0, 0, 0, 0);
                    if (has_x) xv[w] = *reinterpret_cast<const uint4 *>(xrow + (kb * 16 + 4 * w) * 16);
                }
                mac_word<DT>(acc, cur.wa.x, cur.wb.x, zla, zha, s2a, zlb, zhb, s2b, xv[0]);
                mac_word<DT>(acc2, cur.wa.y, cur.wb.y, zla, zha, s2a, zlb, zhb, s2b, xv[1]);
                mac_word<DT>(acc, cur.wa.z, cur.wb.z, zla, zha, s2a, zlb, zhb, s2b, xv[2]);
                mac_word<DT>(acc2, cur.wa.w, cur.wb.w, zla, zha, s2a, zlb, zhb, s2b, xv[3]);

                if (++kb == nblk) { kb = 0; ++rb; }
            }
        }
    }
    if (n_units > 0) {
        const int last_rb = (kb == 0) ? rb - 1 : rb;
        const int last_kb = (kb == 0) ? nblk - 1 : kb - 1;
        flush(last_rb, last_kb);
    }
    __syncthreads();

    // ---- row blocks split between warps: sum the warps' slots in warp order.
    // Row blocks of this CTA: rb_lo .. rb_hi; warp (rbl % NW) handles rb_lo + rbl.
    const int rb_lo = (int)(cu0 / nblk), rb_hi = (int)((cu1 - 1) / nblk);
    const float *slots = reinterpret_cast<const float *>(smem + L.slots);
    for (int rbl = warp; rbl <= rb_hi - rb_lo && n_cta > 0; rbl += kNW) {
        const int frb = rb_lo + rbl;
        const long long ub0 = (long long)frb * nblk, ub1 = ub0 + nblk;   // the block's units
        // is any warp's piece a partial piece of this block?
        bool any = false;
        for (int w = 0; w < kNW; ++w) {
            const long long a = cu0 + range_start(w, n_cta, kNW), b = cu0 + range_start(w + 1, n_cta, kNW);
            if (a < b && a < ub1 && b > ub0 && !(a <= ub0 && b >= ub1)) any = true;
        }
        if (!any) continue;                       // written directly by its warp
        const bool cta_complete = cu0 <= ub0 && cu1 >= ub1;
        const int side = (frb == rb_lo) ? 0 : 1;
        float *gslot = p.ws + ((size_t)blockIdx.x * 2 + side) * kSlot;
        for (int e = lane; e < kUnitRows * p.M; e += 32) {
            const int r = e / p.M, m = e - (e / p.M) * p.M;
            float sum = 0.f;
            for (int w = 0; w < kNW; ++w) {
                const long long a = cu0 + range_start(w, n_cta, kNW), b = cu0 + range_start(w + 1, n_cta, kNW);
                if (!(a < b && a < ub1 && b > ub0) || (a <= ub0 && b >= ub1)) continue;
                const int wfirst = (int)(a / nblk);
                sum += slots[((size_t)w * 2 + (frb == wfirst ? 0 : 1)) * kSlot + r * 8 + m];
            }
            const int row = frb * kUnitRows + r;
            if (cta_complete) {
                if (row < p.N) p.out[(size_t)m * p.N + row] = f32_to_dt<DT>(sum);
            } else {
                gslot[r * 8 + m] = sum;
            }
        }
        if (cta_complete) continue;
        // ---- split between CTAs: ticket; the last CTA sums every CTA's partial in order
        __threadfence();
        __syncwarp();
        const int cf = cta_of(ub0, p.U, p.C), cl = cta_of(ub1 - 1, p.U, p.C);
        int ticket = 0;
        if (lane == 0) ticket = atomicAdd(p.counters + frb, 1);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket != cl - cf) continue;
        __threadfence();
        for (int e = lane; e < kUnitRows * p.M; e += 32) {
            const int r = e / p.M, m = e - (e / p.M) * p.M;
            float sum = 0.f;
            for (int c = cf; c <= cl; ++c) {
                const int crb_lo = (int)(range_start(c, p.U, p.C) / nblk);
                sum += __ldcg(p.ws + ((size_t)c * 2 + (frb == crb_lo ? 0 : 1)) * kSlot + r * 8 + m);
            }
            const int row = frb * kUnitRows + r;
            if (row < p.N) p.out[(size_t)m * p.N + row] = f32_to_dt<DT>(sum);
        }
        if (lane == 0) p.counters[frb] = 0;
    }
}

}  // namespace sk

// ------------------------------------------------------------------ host side
static int sk_xpitch(int K) {
    const int nblk = (K + sk::kUnitK - 1) / sk::kUnitK;
    int bytes = nblk * 256;
    return ((bytes + 127) / 128) * 128 + 64;   // odd multiple of 64
}

size_t decode_sk_smem_bytes(int M, int K) { return sk::sk_layout(M, sk_xpitch(K)).total; }

size_t decode_sk_workspace_floats(int sm_count) { return (size_t)sm_count * 2 * sk::kSlot; }

bool decode_sk_applicable(int M, int K) { return decode_sk_smem_bytes(M, K) <= 220 * 1024; }

template <int DT, bool ASYM, int NS>
static cudaError_t launch_sk_t(const int32_t *qw, const sk::Params &p, size_t smem, int grid,
                               cudaStream_t s, bool pdl) {
    auto kern = sk::decode_sk_kernel<DT, ASYM, NS>;
    if (smem > 48 * 1024) {
        cudaError_t e = raise_smem_cap(reinterpret_cast<const void *>(kern), smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(sk::kNW * 32, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, qw, p);
}

cudaError_t launch_decode_sk(const GemmArgs &a, int ns, const DeviceInfo &dev, float *ws, int *counters,
                             cudaStream_t s, bool pdl) {
    sk::Params p;
    p.x = (const uint16_t *)a.x;
    p.scales = (const uint16_t *)a.scales;
    p.qz = a.qzeros;
    p.out = (uint16_t *)a.out;
    p.ws = ws;
    p.counters = counters;
    p.status = dev.status;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = a.G;
    p.ng = a.K / a.G;
    p.log2G = a.G == 32 ? 5 : (a.G == 64 ? 6 : 7);
    p.nblk = (a.K + sk::kUnitK - 1) / sk::kUnitK;
    p.xpitch = sk_xpitch(a.K);
    const int rblocks = (a.N + sk::kUnitRows - 1) / sk::kUnitRows;
    p.U = (long long)rblocks * p.nblk;
    int grid = dev.sm_count;
    if ((long long)grid > p.U) grid = (int)p.U;
    p.C = grid;
    const bool asym = a.qzeros != nullptr;
    const size_t smem = decode_sk_smem_bytes(a.M, a.K);
#define W4A16_SK_LAUNCH(NSV)                                                                      \
    if (a.dtype == 0)                                                                             \
        return asym ? launch_sk_t<0, true, NSV>(a.qweight, p, smem, grid, s, pdl)                  \
                    : launch_sk_t<0, false, NSV>(a.qweight, p, smem, grid, s, pdl);                \
    return asym ? launch_sk_t<1, true, NSV>(a.qweight, p, smem, grid, s, pdl)                      \
                : launch_sk_t<1, false, NSV>(a.qweight, p, smem, grid, s, pdl);
    if (ns == 2) { W4A16_SK_LAUNCH(2) }
    if (ns == 4) { W4A16_SK_LAUNCH(4) }
    W4A16_SK_LAUNCH(6)
#undef W4A16_SK_LAUNCH
}

}  // namespace w4a16
