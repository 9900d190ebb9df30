// prefill.cu -- fused-dequant W4A16 GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA, sm_103a).
//
// "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP skinny
// decode", PR description: batch sizes above the decode threshold go to a
// fused dequant GEMM (optimised for prefill / batched inference) that reads
// the same packed [N, K/8] weights.
//
// Design (GB300-first):
//  * One CTA computes a 256 (weight rows n) x BN (tokens m) output tile as
//    two 128-row halves.  The dequantised weights are the MMA's A operand
//    (M = 128 per half) and the activations the shared B operand (N = BN <=
//    256): every x tile feeds 2 x 128 x BN MACs per k, which halves the
//    L2 -> SM activation traffic per FLOP against a 128-row tile.
//  * Warps 0 and 3: TMA producers, one issuing thread each (a thread's TMA
//    boxes are issued one after another, so two issuers keep more bytes in
//    flight).  Warp 0 loads, per 64-wide K step, the x tile (BN rows x
//    128 B, 128-byte swizzle) into an SX-deep ring; warp 3 loads the packed
//    weights of 256 k at a time (256 rows x 128 B, 128-byte swizzle) into an
//    SW-deep ring.
//  * Warps 4..11: dequantisers, one weight row per thread.  Each turns its
//    row's 32 packed bytes per step into 64 bf16/fp16 weights in the
//    canonical K-major 128-byte-swizzled layout the tensor core reads, fences
//    them into the async proxy, and each warp arrives once on the A-ring
//    barrier.  Scales and zero points come one packed-weight tile ahead, one
//    vector load per tile, issued after the tile's first arrive (an arrive
//    has release semantics and would otherwise wait for the loads to land).
//    After the main loop the same warps are the epilogue:
//    tcgen05.ld from TMEM (lane quadrant = warp % 4), the optional bias of
//    the row added, one rounding to the output dtype, a [BN x 256] tile
//    staged in shared memory, one TMA store.
//  * Warp 1: TMEM allocation (512 columns: two fp32 accumulators) and the
//    single-thread MMA issuer (tcgen05.mma.cta_group::1.kind::f16,
//    128 x BN x 16 per instruction, two per 16 k); tcgen05.commit releases
//    ring slots and finally signals the epilogue.
//  * Few output tiles (small M): K is split over a thread-block cluster of
//    KS <= 8 CTAs, rank r taking packed-weight tiles [r T / KS, (r+1) T / KS)
//    of the T along K into its own TMEM accumulator.  The fp32 partial tiles
//    are laid over the idle rings and summed in rank order through
//    distributed shared memory, rank r storing token rows [r BN / KS,
//    (r + 1) BN / KS) of the tile (deterministic; KS = 1 is the plain path).
//    The host picks BN and KS with a time model fitted to this kernel and
//    the GPU's cluster occupancy.
//  * Swapped form (128-token tiles): x is the MMA's A operand (M = 128
//    tokens) and the tile's 256 dequantised weight rows are B (N = 256), one
//    MMA per 16 k instead of two; TMEM lanes are then tokens, and the
//    epilogue stages y in four 64-row blocks with a 128-byte swizzle.
//  * Row split: when the wide tiles leave a last wave partly empty, the host
//    may run the weight rows as two launches -- the rows that fill whole
//    waves of wide tiles, then the rest with a configuration of their own
//    (often a K split) -- writing two column blocks of y (out row stride
//    `ldo`).
//  * Dense form (the dequantised prefill cache): the weight operand is a
//    dtype matrix W [N, K] already holding RN((q - z) s); warp 3 loads its
//    64-k steps (two 128-row boxes, 128-byte swizzle: exactly the canonical
//    layout the dequantisers would write) straight into the A ring, and
//    warps 4..11 only run the epilogue.
//  * Every mbarrier wait is bounded (%globaltimer); a wait that runs out sets
//    the device status word and a CTA abort flag, and every role leaves its
//    loop, so the CTA still frees its TMEM and exits.
#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"

#include <algorithm>
#include <type_traits>
#include <cooperative_groups.h>
#include <cuda.h>

namespace w4a16 {

constexpr int kHalf = 128;                     // rows per MMA (M)
constexpr int kBW = 2 * kHalf;                 // weight rows per CTA
constexpr int kBK = 64;                        // k per MMA step
constexpr int kWK = 256;                       // k per packed-weight stage (128 B a row)
constexpr int kStepsPerW = kWK / kBK;          // 4
constexpr int kThreads = 384;                  // 12 warps
constexpr int kDeqWarps = 8;
constexpr int kATileBytes = kBW * kBK * 2;     // 32 KB: both halves
constexpr int kWTileBytes = kBW * kWK / 2;     // 32 KB packed

struct PrefillParams {
    DqConsts dq;          // dequantiser masks / magics, passed as data (see dequant.cuh)
    const uint16_t *scales;
    const int32_t *qz;
    uint16_t *out;        // y [M, N] (written directly when K is split; else by TMA store)
    const uint16_t *bias; // [N] added before the rounding, or null
    int M, N, K, G, ng;
    int BN, SX, SA, SW;
    int n_mtiles;
    int KS;               // CTAs of a cluster splitting K (1 = no split)
    int ldo;              // elements between rows of out (N, or more for a block of columns)
    int swap;             // 1: x is the MMA's A operand (128 tokens), the weights B (N = 256); BN = 128
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

template <int DT>
__device__ __forceinline__ float dt16_to_f32(uint16_t v) {
    if (DT == 0) return __half2float(__ushort_as_half(v));
    return __bfloat162float(__ushort_as_bfloat16(v));
}

struct SmemLayout {
    uint32_t x_off, a_off, w_off, bar_off, total;
};

__host__ __device__ inline SmemLayout prefill_layout(int BN, int SX, int SA, int SW) {
    SmemLayout L;
    uint32_t off = 0;
    L.x_off = off;
    off += (uint32_t)SX * BN * 128;
    off = (off + 1023u) & ~1023u;
    L.a_off = off;
    off += (uint32_t)SA * kATileBytes;
    L.w_off = off;
    off += (uint32_t)SW * kWTileBytes;
    L.bar_off = off;
    off += (uint32_t)(2 * SX + 2 * SA + 2 * SW + 1) * 8 + 16;
    L.total = off + 1024;  // slack for aligning the dynamic base to 1024
    return L;
}

// One 64-k step of MMAs from descriptor words.  The issuing thread's
// instruction stream sets the pace of a step, so the descriptors are built
// once per step rather than per MMA (about 1 % on the Llama layers at
// M >= 512): the low word of a shared-memory descriptor (smem_desc_sw128)
// is (address >> 4) plus fixed fields, so the 16-k slice kk of a 128-byte-
// swizzled operand is lo + 2 kk, and the high word is the same for every
// operand.  first = 0 starts a fresh accumulation with the step's first MMA
// (predicate p); the others accumulate (predicate q, true because an
// instruction descriptor is never zero).
// tc_mma8: the plain form, weight halves a0 / a1 (A) against x (B), into
// the accumulators at d and d + 256.
__device__ __forceinline__ void tc_mma8(uint32_t d, uint32_t a0lo, uint32_t a1lo, uint32_t blo, uint32_t hi,
                                        uint32_t idesc, uint32_t first) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 a, b;\n\t.reg .b32 t;\n\t"
        "setp.ne.b32 p, %6, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "mov.b64 a, {%1, %4};\n\tmov.b64 b, {%3, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n\t"
        "mov.b64 a, {%2, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%7], a, b, %5, p;\n\t"
        "add.u32 t, %1, 2;\n\tmov.b64 a, {t, %4};\n\tadd.u32 t, %3, 2;\n\tmov.b64 b, {t, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, q;\n\t"
        "add.u32 t, %2, 2;\n\tmov.b64 a, {t, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%7], a, b, %5, q;\n\t"
        "add.u32 t, %1, 4;\n\tmov.b64 a, {t, %4};\n\tadd.u32 t, %3, 4;\n\tmov.b64 b, {t, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, q;\n\t"
        "add.u32 t, %2, 4;\n\tmov.b64 a, {t, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%7], a, b, %5, q;\n\t"
        "add.u32 t, %1, 6;\n\tmov.b64 a, {t, %4};\n\tadd.u32 t, %3, 6;\n\tmov.b64 b, {t, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, q;\n\t"
        "add.u32 t, %2, 6;\n\tmov.b64 a, {t, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%7], a, b, %5, q;\n\t}"
        ::"r"(d), "r"(a0lo), "r"(a1lo), "r"(blo), "r"(hi), "r"(idesc), "r"(first), "r"(d + 256u)
        : "memory");
}

// tc_mma4_swp: the swapped form, x (A, 128 tokens) against all 256 weight
// rows (B), into the accumulator at d.
__device__ __forceinline__ void tc_mma4_swp(uint32_t d, uint32_t xlo, uint32_t wlo, uint32_t hi, uint32_t idesc,
                                            uint32_t first) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 a, b;\n\t.reg .b32 t;\n\t"
        "setp.ne.b32 p, %5, 0;\n\tsetp.ne.b32 q, %4, 0;\n\t"
        "mov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, p;\n\t"
        "add.u32 t, %1, 2;\n\tmov.b64 a, {t, %3};\n\tadd.u32 t, %2, 2;\n\tmov.b64 b, {t, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, q;\n\t"
        "add.u32 t, %1, 4;\n\tmov.b64 a, {t, %3};\n\tadd.u32 t, %2, 4;\n\tmov.b64 b, {t, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, q;\n\t"
        "add.u32 t, %1, 6;\n\tmov.b64 a, {t, %3};\n\tadd.u32 t, %2, 6;\n\tmov.b64 b, {t, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, q;\n\t}"
        ::"r"(d), "r"(xlo), "r"(wlo), "r"(hi), "r"(idesc), "r"(first)
        : "memory");
}

// Position in a ring of mbarrier-guarded slots: the slot and the parity of
// its current phase, advanced by one per use.  (Counters instead of i % S and
// i / S: with the ring depths as launch parameters those are integer
// divisions, and on the MMA issuer's and the dequantisers' per-step paths
// they cost about a fifth of the step.)
struct RingPos {
    int slot = 0;
    uint32_t phase = 0u;
    __device__ __forceinline__ void next(int depth) {
        if (++slot == depth) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// The epilogue stages a [BN][256] output tile (512 B a row) over the x and A rings.
__host__ __device__ inline bool prefill_epilogue_fits(int BN, int SX, int SA) {
    return (uint32_t)BN * kBW * 2 <= (uint32_t)SX * BN * 128 + (uint32_t)SA * kATileBytes;
}

template <int DT, bool ASYM, bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_out, const PrefillParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const SmemLayout L = prefill_layout(p.BN, p.SX, p.SA, p.SW);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int SX = p.SX, SA = p.SA, SW = p.SW;

    // With KS > 1 the KS CTAs of a cluster share one output tile, rank r
    // taking packed-weight tiles [r nwt / KS, (r + 1) nwt / KS) of K.
    const int KS = p.KS;
    const int krank = KS > 1 ? (int)cluster_ctarank() : 0;
    const int tile = (int)blockIdx.x / KS;
    const int mt = tile % p.n_mtiles;
    const int nt = tile / p.n_mtiles;
    const int m0 = mt * p.BN, n0 = nt * kBW;
    const int nk_all = (p.K + kBK - 1) / kBK;
    const int nwt = (p.K + kWK - 1) / kWK;           // packed-weight tiles along K
    const int js0 = (int)((long long)krank * nwt / KS), js1 = (int)((long long)(krank + 1) * nwt / KS);
    const int is0 = js0 * kStepsPerW;                // first 64-k step of this CTA
    const int nk = min(js1 * kStepsPerW, nk_all) - is0;   // steps of this CTA

    const uint32_t bar_base = smem_u32(smem + L.bar_off);
    auto xfull = [&](int s) { return bar_base + 8u * s; };
    auto xempty = [&](int s) { return bar_base + 8u * (SX + s); };
    auto afull = [&](int a) { return bar_base + 8u * (2 * SX + a); };
    auto aempty = [&](int a) { return bar_base + 8u * (2 * SX + SA + a); };
    auto wfull = [&](int w) { return bar_base + 8u * (2 * SX + 2 * SA + w); };
    auto wempty = [&](int w) { return bar_base + 8u * (2 * SX + 2 * SA + SW + w); };
    const uint32_t acc_bar = bar_base + 8u * (2 * SX + 2 * SA + 2 * SW);
    uint32_t *tmem_slot =
        reinterpret_cast<uint32_t *>(smem + L.bar_off + 8 * (2 * SX + 2 * SA + 2 * SW + 1));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t x_base = smem_u32(smem + L.x_off);
    const uint32_t a_base = smem_u32(smem + L.a_off);
    const uint32_t w_base = smem_u32(smem + L.w_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull(s), 1);
            mbar_init(xempty(s), 1);             // MMA commit
        }
        for (int a = 0; a < SA; ++a) {
            mbar_init(afull(a), DENSE ? 1 : kDeqWarps);   // the TMA's arrive, or one per dequant warp
            mbar_init(aempty(a), 1);             // MMA commit
        }
        for (int w = 0; w < SW; ++w) {
            mbar_init(wfull(w), 1);
            mbar_init(wempty(w), kDeqWarps);
        }
        mbar_init(acc_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_out);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;

    grid_dependents_launch();

    if (warp == 0) {
        // ------------------------------------------------------------ x producer
        if (lane == 0) {
            grid_dependency_wait();  // x may be written by the previous kernel
            const uint32_t xtx = (uint32_t)p.BN * 128u;
            RingPos r;
            for (int i = 0; i < nk; ++i, r.next(SX)) {
                if (!mbar_wait_bounded(xempty(r.slot), r.phase ^ 1u, p.status, abort_flag)) break;
                mbar_arrive_expect_tx(xfull(r.slot), xtx);
                tma_load_2d(x_base + (uint32_t)r.slot * p.BN * 128u, &tmap_x, xfull(r.slot), (is0 + i) * kBK, m0);
            }
        }
    } else if (warp == 3 && DENSE) {
        // ------------------------------------------------------------ dense weight producer
        // 64-k steps of the dtype weight cache straight into the A ring.
        if (lane == 0) {
            RingPos r;
            for (int i = 0; i < nk; ++i, r.next(SA)) {
                if (!mbar_wait_bounded(aempty(r.slot), r.phase ^ 1u, p.status, abort_flag)) break;
                mbar_arrive_expect_tx(afull(r.slot), (uint32_t)kATileBytes);
                const uint32_t dst = a_base + (uint32_t)r.slot * kATileBytes;
                tma_load_2d(dst, &tmap_w, afull(r.slot), (is0 + i) * kBK, n0);
                tma_load_2d(dst + kHalf * 128u, &tmap_w, afull(r.slot), (is0 + i) * kBK, n0 + kHalf);
            }
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ weight producer
        // (its own issuing thread: one thread's TMA boxes complete one after another)
        if (lane == 0) {
            const int nw = js1 - js0;
            RingPos r;
            for (int j = 0; j < nw; ++j, r.next(SW)) {
                if (!mbar_wait_bounded(wempty(r.slot), r.phase ^ 1u, p.status, abort_flag)) break;
                mbar_arrive_expect_tx(wfull(r.slot), (uint32_t)kWTileBytes);
                tma_load_2d(w_base + (uint32_t)r.slot * kWTileBytes, &tmap_w, wfull(r.slot), (js0 + j) * (kWK / 8),
                            n0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // Plain: two 128 x BN x 16 MMAs per 16 k (weight halves as A, x as
            // B).  Swapped (BN = 128): one 128 x 256 x 16 MMA, x as A and all
            // 256 weight rows as B -- half the instructions for the same tile,
            // each MMA costing about the same at any N.  The two forms are
            // separate loops: this thread's instruction stream sets the pace
            // of the step, and a per-MMA branch measured ~6 % slower.
            auto issue_steps = [&](auto swap_tag) {
                constexpr bool SWP = decltype(swap_tag)::value;
                const uint32_t idesc = SWP ? make_idesc_f16(DT, kHalf, kBW) : make_idesc_f16(DT, kHalf, p.BN);
                const uint32_t dlo0 = (uint32_t)smem_desc_sw128(0u), dhi = (uint32_t)(smem_desc_sw128(0u) >> 32);
                RingPos rx, ra;
                for (int i = 0; i < nk; ++i, rx.next(SX), ra.next(SA)) {
                    const int s = rx.slot, a = ra.slot;
                    if (!mbar_wait_bounded(xfull(s), rx.phase, p.status, abort_flag)) break;
                    if (!mbar_wait_bounded(afull(a), ra.phase, p.status, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t xa = x_base + (uint32_t)s * p.BN * 128u;
                    const uint32_t aa = a_base + (uint32_t)a * kATileBytes;
                    {
                        const uint32_t xlo = dlo0 + (xa >> 4), alo = dlo0 + (aa >> 4);
                        const uint32_t first = i > 0 ? 1u : 0u;
                        if constexpr (SWP) {
                            tc_mma4_swp(tmem_d, xlo, alo, dhi, idesc, first);
                        } else {
                            tc_mma8(tmem_d, alo, alo + (uint32_t)(kHalf * 128 / 16), xlo, dhi, idesc, first);
                        }
                    }
                    tc_commit(xempty(s));
                    tc_commit(aempty(a));
                }
            };
            if (p.swap)
                issue_steps(std::true_type{});
            else
                issue_steps(std::false_type{});
            tc_commit(acc_bar);
        }
        __syncwarp();
    } else if (warp >= 4) {
        bool ok = true;
        if constexpr (!DENSE) {
        // ------------------------------------------------------------ dequantisers
        const int r = threadIdx.x - 128;               // weight row within the tile, 0..255
        const int n = n0 + r;
        const bool vrow = n < p.N;
        const int zshift = 4 * (n & 7);
        // Scales and zero points: the groups of one packed-weight tile (256 k)
        // for this row are fetched with one vector load each (K a multiple
        // of 256 keeps them aligned; else one load per group), one tile
        // ahead, right after the tile's first A-ring arrive -- so that the
        // loads neither sit behind the dequantiser's shared-memory stores
        // every step nor hold up a release-arrive while they are in flight.
        // At the start of a tile they are unpacked into per-step registers.
        const int gcount = kWK / p.G;                  // groups per tile: 8, 4 or 2
        const bool vec_meta = (p.K % kWK) == 0;
        uint32_t vs[4], vz[8];
        auto load_tile_meta = [&](int j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) vs[e] = 0u;
#pragma unroll
            for (int e = 0; e < 8; ++e) vz[e] = 0u;
            if (!vrow || j * kWK >= p.K) return;
            const int gA = j * gcount;
            const uint16_t *sp = p.scales + (size_t)n * p.ng + gA;
            const int32_t *zp = ASYM ? p.qz + (size_t)(n >> 3) * p.ng + gA : nullptr;
            if (vec_meta) {
                if (gcount == 8) {
                    const uint4 v = ldg_nc_v4(sp);
                    vs[0] = v.x; vs[1] = v.y; vs[2] = v.z; vs[3] = v.w;
                    if (ASYM) {
                        const uint4 z0 = ldg_nc_v4(zp), z1 = ldg_nc_v4(zp + 4);
                        vz[0] = z0.x; vz[1] = z0.y; vz[2] = z0.z; vz[3] = z0.w;
                        vz[4] = z1.x; vz[5] = z1.y; vz[6] = z1.z; vz[7] = z1.w;
                    }
                } else if (gcount == 4) {
                    const uint2 v = ldg_nc_v2(sp);
                    vs[0] = v.x; vs[1] = v.y;
                    if (ASYM) {
                        const uint4 z0 = ldg_nc_v4(zp);
                        vz[0] = z0.x; vz[1] = z0.y; vz[2] = z0.z; vz[3] = z0.w;
                    }
                } else {
                    vs[0] = ldg_nc_u32(sp);
                    if (ASYM) {
                        const uint2 z0 = ldg_nc_v2(zp);
                        vz[0] = z0.x; vz[1] = z0.y;
                    }
                }
            } else {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    if (g < gcount && gA + g < p.ng) {
                        const uint32_t h = __ldg(sp + g);
                        vs[g >> 1] |= (g & 1) ? (h << 16) : h;
                        if (ASYM) vz[g] = (uint32_t)__ldg(zp + g);
                    }
                }
            }
        };
        // per-step (k and k + 32 halves of each 64-wide step) scale and zero word
        uint32_t rs_lo[kStepsPerW], rs_hi[kStepsPerW], rz_lo[kStepsPerW], rz_hi[kStepsPerW];
        auto unpack_tile_meta = [&]() {
#pragma unroll
            for (int jj = 0; jj < kStepsPerW; ++jj) {
                if (gcount == 8) {          // G = 32: groups 2jj, 2jj + 1
                    rs_lo[jj] = vs[jj] & 0xFFFFu;
                    rs_hi[jj] = vs[jj] >> 16;
                    rz_lo[jj] = vz[2 * jj];
                    rz_hi[jj] = vz[2 * jj + 1];
                } else if (gcount == 4) {   // G = 64: group jj
                    rs_lo[jj] = rs_hi[jj] = (jj & 1) ? (vs[jj >> 1] >> 16) : (vs[jj >> 1] & 0xFFFFu);
                    rz_lo[jj] = rz_hi[jj] = vz[jj];
                } else {                    // G = 128: group jj / 2
                    rs_lo[jj] = rs_hi[jj] = (jj >> 1) ? (vs[0] >> 16) : (vs[0] & 0xFFFFu);
                    rz_lo[jj] = rz_hi[jj] = vz[jj >> 1];
                }
            }
        };
        load_tile_meta(js0);

        // A tile (both halves): half h = r / 128 at h * 16 KB; 128-byte rows,
        // 16-byte chunk c of row r at position c ^ (r % 8) within its 8-row atom.
        const uint32_t sw = (uint32_t)(r & 7);
        const uint32_t a_row = (uint32_t)(r >> 7) * (kHalf * 128) + (uint32_t)((r & 127) >> 3) * 1024u +
                               sw * 128u;
        const uint32_t w_row = (uint32_t)(r >> 3) * 1024u + sw * 128u;   // packed tile, same swizzle
        const DqConsts dc = p.dq;
        // G >= 64: both 32-k halves of a step are in one group, so its constants
        // are built once (the dequantisers share the SM's issue slots with the
        // MMA issuer: 1-2.5 % on the Llama layers at M = 1920).
        const int one_group = gcount <= 4 ? 1 : 0;
        RingPos rw, ra;                                // packed-weight and A ring positions
        for (int i0 = 0; i0 < nk && ok; i0 += kStepsPerW) {
            unpack_tile_meta();
#pragma unroll
            for (int d = 0; d < kStepsPerW; ++d) {
                const int i = i0 + d;
                if (i < nk && ok) {
                    const uint32_t slo = rs_lo[d];
                    uint32_t zlo = 8u;
                    if (ASYM) zlo = (rz_lo[d] >> zshift) & 0xFu;
                    const int jj = d, swi = rw.slot;
                    if (jj == 0 && !mbar_wait_bounded(wfull(swi), rw.phase, p.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const unsigned char *wrow = smem + L.w_off + (size_t)swi * kWTileBytes + w_row;
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(wrow + (((uint32_t)(2 * jj) ^ sw) << 4));
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(wrow + (((uint32_t)(2 * jj + 1) ^ sw) << 4));
                    if (jj == kStepsPerW - 1 || i == nk - 1) {
                        // Release the packed-weight slot only once this
                        // thread's loads from it have returned (the asm
                        // consumes the loaded registers) and are ordered
                        // before the async-proxy copy that will refill it.
                        asm volatile("" ::"r"(w0.x), "r"(w0.y), "r"(w0.z), "r"(w0.w), "r"(w1.x), "r"(w1.y),
                                     "r"(w1.z), "r"(w1.w)
                                     : "memory");
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(wempty(swi));
                        rw.next(SW);
                    }
                    const int a = ra.slot;
                    const uint32_t aph = ra.phase;
                    ra.next(SA);
                    if (!mbar_wait_bounded(aempty(a), aph ^ 1u, p.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t zc_lo = zseq2<DT>(zlo), s2lo = rep2(slo);
                    uint32_t zc_hi = zc_lo, s2hi = s2lo;
                    if (one_group == 0) {        // G = 32: the step's two halves have their own group
                        zc_hi = zseq2<DT>(ASYM ? (rz_hi[d] >> zshift) & 0xFu : 8u);
                        s2hi = rep2(rs_hi[d]);
                    }
                    unsigned char *adst = smem + L.a_off + (size_t)a * kATileBytes + a_row;
                    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[4];
                        dq_word_seq_rt<DT>(words[c], dc, c < 4 ? zc_lo : zc_hi, c < 4 ? s2lo : s2hi, o);
                        *reinterpret_cast<uint4 *>(adst + (((uint32_t)c ^ sw) << 4)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    fence_proxy_async_smem();   // each writer: generic -> async proxy
                    __syncwarp();
                    if (lane == 0) mbar_arrive(afull(a));
                    if (d == 0 && js0 + i / kStepsPerW + 1 < js1) load_tile_meta(js0 + i / kStepsPerW + 1);
                }
            }
        }
        }   // !DENSE

        // ------------------------------------------------------------ epilogue
        const bool have_acc = ok && mbar_wait_bounded(acc_bar, 0u, p.status, abort_flag);
        if (KS > 1) {
            // K split: this CTA's fp32 partial tile -> part[token][weight row]
            // over the (idle) rings; summed across the cluster below.
            if (have_acc && p.swap) {
                // TMEM lane = token, column = weight row.  Each thread writes 16
                // consecutive weight rows of its token as four 16-byte chunks,
                // chunk ch of token row c stored at ch ^ (c % 8) (a quarter-warp
                // then hits eight different bank groups); the sum below reads
                // with the same permutation.
                tc_fence_after();
                const int q = warp & 3, h = (warp - 4) >> 2;
                const int c = 32 * q + lane;                          // token row of the tile
                const uint32_t tbase = tmem_d + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * kHalf);
                float4 *prow = reinterpret_cast<float4 *>(smem) + (size_t)c * (kBW / 4);
                for (int c0 = 0; c0 < kHalf; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tbase + (uint32_t)c0, v);
                    const int ch0 = (h * kHalf + c0) >> 2;
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        prow[(ch0 + u) ^ (c & 7)] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                                                __uint_as_float(v[4 * u + 2]),
                                                                __uint_as_float(v[4 * u + 3]));
                }
            } else if (have_acc) {
                tc_fence_after();
                const int q = warp & 3, h = (warp - 4) >> 2;
                const int nl = h * kHalf + 32 * q + lane;
                const uint32_t tbase = tmem_d + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * 256);
                float *part = reinterpret_cast<float *>(smem);
                for (int c0 = 0; c0 < p.BN; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tbase + (uint32_t)c0, v);
#pragma unroll
                    for (int jx = 0; jx < 16; ++jx) part[(size_t)(c0 + jx) * kBW + nl] = __uint_as_float(v[jx]);
                }
            }
        } else {
            if (have_acc && p.swap) {
                // TMEM lane = token, column = weight row.  The tile is staged as
                // four blocks of 64 weight rows, [BN tokens][128 B] each in the
                // 128-byte-swizzled layout of the store map (16-byte chunk ch of
                // token row c at ch ^ (c % 8)), and leaves in four TMA stores.
                tc_fence_after();
                const int q = warp & 3, h = (warp - 4) >> 2;
                const int c = 32 * q + lane;                          // token row of the tile
                const uint32_t tbase = tmem_d + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * kHalf);
                for (int c0 = 0; c0 < kHalf; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tbase + (uint32_t)c0, v);
                    const int col = h * kHalf + c0;                   // first weight row of the 16
                    uint32_t pk[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float a = __uint_as_float(v[2 * u]), b = __uint_as_float(v[2 * u + 1]);
                        if (p.bias != nullptr) {
                            const int n = n0 + col + 2 * u;
                            if (n < p.N) a += dt16_to_f32<DT>(__ldg(p.bias + n));
                            if (n + 1 < p.N) b += dt16_to_f32<DT>(__ldg(p.bias + n + 1));
                        }
                        pk[u] = (uint32_t)f32_to_dt16<DT>(a) | ((uint32_t)f32_to_dt16<DT>(b) << 16);
                    }
                    unsigned char *blk = smem + (size_t)(col >> 6) * ((size_t)p.BN * 128) + (size_t)c * 128;
                    const int ch = (col & 63) >> 3;                   // two 16-byte chunks of 8 weight rows
                    *reinterpret_cast<uint4 *>(blk + (((ch) ^ (c & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4 *>(blk + (((ch + 1) ^ (c & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
                fence_proxy_async_smem();
            } else if (have_acc) {
                tc_fence_after();
                const int q = warp & 3, h = (warp - 4) >> 2;
                const int nl = h * kHalf + 32 * q + lane;            // row of the tile
                const uint32_t tbase = tmem_d + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * 256);
                uint16_t *stage = reinterpret_cast<uint16_t *>(smem);   // [BN][256], over x/A rings
                const float bv = (p.bias != nullptr && n0 + nl < p.N) ? dt16_to_f32<DT>(p.bias[n0 + nl]) : 0.f;
                for (int c0 = 0; c0 < p.BN; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tbase + (uint32_t)c0, v);
#pragma unroll
                    for (int jx = 0; jx < 16; ++jx)
                        stage[(size_t)(c0 + jx) * kBW + nl] = f32_to_dt16<DT>(__uint_as_float(v[jx]) + bv);
                }
                fence_proxy_async_smem();
            }
            named_barrier_sync(1, kDeqWarps * 32);
            if (have_acc && threadIdx.x == 128) {
                if (p.swap) {
                    for (int b = 0; b < kBW / 64; ++b)
                        if (n0 + 64 * b < p.N)   // boxes wholly past the last weight row are not issued
                            tma_store_2d(&tmap_out, smem_u32(smem) + (uint32_t)(b * p.BN * 128), n0 + 64 * b, m0);
                } else {
                    tma_store_2d(&tmap_out, smem_u32(smem), n0, m0);
                }
                bulk_commit_group();
                bulk_wait_group_all();
            }
        }
    }

    if (KS > 1) {
        // Sum the KS partial tiles in rank order (deterministic); rank r
        // writes token rows [r BN / KS, (r + 1) BN / KS) of the tile.
        cluster_sync_all();
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        float *part = reinterpret_cast<float *>(smem);
        const float *peer[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) peer[q] = cluster.map_shared_rank(part, q < KS ? q : 0);
        const int c_lo = (int)((long long)krank * p.BN / KS), c_hi = (int)((long long)(krank + 1) * p.BN / KS);
        const int n_v = (c_hi - c_lo) * (kBW / 4);      // float4 groups of this CTA's rows
        const bool vec_out = (p.ldo & 3) == 0;
        for (int idx = threadIdx.x; idx < n_v; idx += kThreads) {
            const int c = c_lo + (idx >> 6), nl = (idx & 63) * 4;
            const int m = m0 + c, n = n0 + nl;
            if (m >= p.M || n >= p.N) continue;
            const size_t off = (size_t)c * kBW + (p.swap ? (size_t)((((nl >> 2) ^ (c & 7))) << 2) : (size_t)nl);
            float4 sum = *reinterpret_cast<const float4 *>(peer[0] + off);
#pragma unroll
            for (int q = 1; q < 8; ++q) {
                if (q < KS) {
                    const float4 t = *reinterpret_cast<const float4 *>(peer[q] + off);
                    sum.x += t.x; sum.y += t.y; sum.z += t.z; sum.w += t.w;
                }
            }
            if (p.bias != nullptr) {
                sum.x += dt16_to_f32<DT>(p.bias[n]);
                if (n + 1 < p.N) sum.y += dt16_to_f32<DT>(p.bias[n + 1]);
                if (n + 2 < p.N) sum.z += dt16_to_f32<DT>(p.bias[n + 2]);
                if (n + 3 < p.N) sum.w += dt16_to_f32<DT>(p.bias[n + 3]);
            }
            const uint16_t o0 = f32_to_dt16<DT>(sum.x), o1 = f32_to_dt16<DT>(sum.y);
            const uint16_t o2 = f32_to_dt16<DT>(sum.z), o3 = f32_to_dt16<DT>(sum.w);
            uint16_t *dst = p.out + (size_t)m * p.ldo + n;
            if (vec_out && n + 3 < p.N) {
                *reinterpret_cast<uint2 *>(dst) = make_uint2(o0 | ((uint32_t)o1 << 16), o2 | ((uint32_t)o3 << 16));
            } else {
                dst[0] = o0;
                if (n + 1 < p.N) dst[1] = o1;
                if (n + 2 < p.N) dst[2] = o2;
                if (n + 3 < p.N) dst[3] = o3;
            }
        }
        cluster_sync_all();   // keep this CTA's partials alive while the others read them
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_d, 512u);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static bool prefill_cfg_fits(const PrefillCfg &c) {
    return prefill_layout(c.BN, c.stages, c.astages, c.wstages).total <= 227 * 1024 &&
           prefill_epilogue_fits(c.BN, c.stages, c.astages);
}

// A K split sums fp32 partial tiles ([BN][256], 1 KB a token) laid over the rings.
static bool prefill_split_fits(const PrefillCfg &c) {
    return (size_t)c.BN * kBW * 4 <= prefill_layout(c.BN, c.stages, c.astages, c.wstages).bar_off;
}

// Time model of one launch (microseconds, fitted to GB300 timings of this
// kernel over BN x K split x ring depth on the Llama-3.1-8B layers at
// M = 16...1920, median error 1 %, at most 13 %): a CTA spends about
// 2.36 + 0.0014 BN per 256-k packed-weight tile, 3.66 more for start-up,
// pipeline fill and epilogue, and, when K is split, 1.6 + 0.034 BN for the
// cluster reduction.  CTAs run in waves of what fits on the GPU at once: one
// CTA per SM, and with a K split whole clusters of KS CTAs, as many as the
// occupancy query allowed.  (The fit also has 5.5 per launch, the same for
// every choice, so it is left out.)
static double prefill_cost(int bn, int ks, long long tiles, int nwt, const DeviceInfo &dev) {
    const int resident = dev.prefill_clusters[ks];
    if (resident <= 0) return 1e30;
    const long long waves = (tiles + resident - 1) / resident;
    const int per_cta = (nwt + ks - 1) / ks;
    const double t = per_cta * (2.36 + 0.0014 * bn) + 3.66 + (ks > 1 ? 1.6 + 0.034 * bn : 0.0);
    return (double)waves * t;
}

// x beyond this size is streamed from HBM by each wave rather than re-read
// from L2, so its copies take longer to return.
constexpr long long kXHotBytes = 32ll << 20;

// Ring depths for a tile: the dequantised-weight (A) ring three deep, so that
// the dequantisers of a step do not wait for the MMAs of the step before the
// last, with the deepest x ring that still fits.  An x ring of two is enough
// only while x stays in L2; for a larger x the A ring stays two deep and the
// x ring takes the room.  (Measured on the Llama layers: three A stages are
// 1-7 % faster everywhere except an x ring of two over a 55 MB x, 4-15 %
// slower.)
static bool prefill_fit_stages(PrefillCfg &c, long long x_bytes) {
    for (int sa = 3; sa >= 2; --sa) {
        c.astages = sa;
        for (int sx = 6; sx >= 2; --sx) {
            c.stages = sx;
            if (!prefill_cfg_fits(c) || (c.ks > 1 && !prefill_split_fits(c))) continue;
            if (sa == 3 && sx < 3 && x_bytes > kXHotBytes) break;
            return true;
        }
    }
    return false;
}

static int prefill_best_ks(const PrefillCfg &base, long long tiles, int nwt, const DeviceInfo &dev, double *cost) {
    int best = 1;
    double best_cost = 1e30;
    for (int ks = 1; ks <= 8 && ks <= nwt; ++ks) {
        PrefillCfg c = base;
        c.ks = ks;
        if (ks > 1 && !prefill_split_fits(c)) continue;
        const double t = prefill_cost(c.BN, ks, tiles, nwt, dev);
        if (t < best_cost * 0.995) {
            best_cost = t;
            best = ks;
        }
    }
    if (cost) *cost = best_cost;
    return best;
}

// Pick BN (tokens per tile, at most M rounded up to 16) and the K split that
// minimise the modelled time, then the ring depths for that split.
PrefillCfg prefill_pick_cfg(int M, int N, int K, int G, int sym, int dtype, const DeviceInfo &dev) {
    (void)G; (void)sym; (void)dtype;
    const int ntiles_n = (N + kBW - 1) / kBW;
    const int nwt = (K + kWK - 1) / kWK;
    const long long xb = (long long)M * K * 2;
    const int bn_max = std::min(256, std::max(16, (M + 15) / 16 * 16));
    PrefillCfg best{bn_max, 2, 2, 2, 1};
    double best_cost = 1e30;
    for (int bn = 16; bn <= bn_max; bn += 16) {
        PrefillCfg c{bn, 2, 2, 2, 1};
        if (!prefill_fit_stages(c, xb)) continue;
        const long long tiles = (long long)((M + bn - 1) / bn) * ntiles_n;
        double t = 0.0;
        // the split needs room for the partial tile over the rings
        PrefillCfg cs = c;
        cs.ks = 2;
        const bool can_split = prefill_fit_stages(cs, xb);
        c.ks = can_split ? prefill_best_ks(cs, tiles, nwt, dev, &t) : 1;
        if (!can_split) t = prefill_cost(bn, 1, tiles, nwt, dev);
        if (t < best_cost * 0.995) {
            best_cost = t;
            best = c;
        }
    }
    prefill_fit_stages(best, xb);
    // 128-token tiles run with swapped operands where that measured faster
    // (5-10 % at a K split of 1 to 3 on the Llama layers at M = 16..1920;
    // mixed at 4 and more).
    if (best.BN == kHalf && best.ks <= 3) best.swap = 1;
    return best;
}

// Per launch, on top of prefill_cost: the constant of the same fit.
constexpr double kLaunchUs = 5.5;

static double prefill_dense_cost(int bn, int ks, long long tiles, int K, const DeviceInfo &dev);
static bool prefill_dense_fit_stages(PrefillCfg &c);

// Modelled time of one launch with configuration c (fused or dense form).
static double prefill_cfg_cost(const PrefillCfg &c, int M, int N, int K, bool dense, const DeviceInfo &dev) {
    const long long tiles = (long long)((M + c.BN - 1) / c.BN) * ((N + kBW - 1) / kBW);
    const int ks = std::max(1, c.ks);
    return kLaunchUs + (dense ? prefill_dense_cost(c.BN, ks, tiles, K, dev)
                              : prefill_cost(c.BN, ks, tiles, (K + kWK - 1) / kWK, dev));
}

static PrefillCfg pick_cfg(int M, int N, int K, bool dense, const DeviceInfo &dev) {
    return dense ? prefill_dense_pick_cfg(M, N, K, dev) : prefill_pick_cfg(M, N, K, 0, 0, 0, dev);
}

// Wave quantisation: with T tiles on R resident CTAs a last, partly filled
// wave costs as much as a full one, and a K split needs a partial tile that
// fits in shared memory (BN <= 208), so it cannot rescue the widest tiles.
// Each tcgen05 MMA takes about as long at N = 160 as at 256, so narrowing
// the tiles to even out the waves wastes tensor throughput instead.  The
// plan may therefore cut the weight rows in two: a first launch of wide
// tiles (K not split) over the rows that fill whole waves, then the
// remaining rows as a second launch with the configuration that suits them
// (often a K split).  The plan with the lower modelled time wins.  The
// same holds for the dense form, with its own configurations and model.
PrefillPlan prefill_pick_plan(int M, int N, int K, bool dense, const DeviceInfo &dev) {
    PrefillPlan plan;
    plan.main = pick_cfg(M, N, K, dense, dev);
    plan.n_split = N;
    plan.tail = plan.main;
    double best = prefill_cfg_cost(plan.main, M, N, K, dense, dev);
    const int resident = dev.prefill_clusters[1];
    const int ntiles_n = (N + kBW - 1) / kBW;
    const long long xb = (long long)M * K * 2;
    const int bn_max = std::min(256, std::max(16, (M + 15) / 16 * 16));
    if (resident <= 0) return plan;
    for (int bn = 16; bn <= bn_max; bn += 16) {
        PrefillCfg c{bn, 2, 2, dense ? 0 : 2, 1};
        if (!(dense ? prefill_dense_fit_stages(c) : prefill_fit_stages(c, xb))) continue;
        if (!dense && bn == kHalf) c.swap = 1;
        const int mt = (M + bn - 1) / bn;
        const int per_wave = resident / mt;            // n-tiles of one full wave
        if (per_wave <= 0) continue;
        const int main_nt = (ntiles_n / per_wave) * per_wave;
        if (main_nt <= 0 || main_nt >= ntiles_n) continue;
        const int n_split = main_nt * kBW;
        const PrefillCfg tail = pick_cfg(M, N - n_split, K, dense, dev);
        const double t = prefill_cfg_cost(c, M, n_split, K, dense, dev) +
                         prefill_cfg_cost(tail, M, N - n_split, K, dense, dev);
        if (t < best * 0.97) {
            best = t;
            plan.main = c;
            plan.n_split = n_split;
            plan.tail = tail;
        }
    }
    return plan;
}

GemmArgs prefill_rows(const GemmArgs &a, int n0, int rows) {
    GemmArgs b = a;
    const size_t ng = a.G > 0 ? (size_t)(a.K / a.G) : 0;
    b.N = rows;
    b.ldo = a.ldo > 0 ? a.ldo : a.N;
    b.out = static_cast<uint16_t *>(a.out) + n0;
    if (a.qweight) b.qweight = a.qweight + (size_t)n0 * (a.K / 8);
    if (a.scales) b.scales = static_cast<const uint16_t *>(a.scales) + (size_t)n0 * ng;
    if (a.qzeros) b.qzeros = a.qzeros + (size_t)(n0 / 8) * ng;
    if (a.bias) b.bias = static_cast<const uint16_t *>(a.bias) + n0;
    if (a.wdense) b.wdense = static_cast<const uint16_t *>(a.wdense) + (size_t)n0 * a.K;
    return b;
}

// ---- dense form (dequantised prefill cache): no packed-weight ring; the x
// and A rings have the same depth.
static bool prefill_dense_fits(const PrefillCfg &c) {
    const SmemLayout L = prefill_layout(c.BN, c.stages, c.astages, 0);
    return L.total <= 227 * 1024 && prefill_epilogue_fits(c.BN, c.stages, c.astages) &&
           (c.ks <= 1 || (size_t)c.BN * kBW * 4 <= L.bar_off);
}

bool prefill_dense_cfg_valid(const PrefillCfg &c) {
    if (c.BN < 16 || c.BN > 256 || c.BN % 16 != 0) return false;
    if (c.swap != 0 && (c.swap != 1 || c.BN != kHalf)) return false;
    if (c.stages < 2 || c.astages < 2) return false;
    if (c.ks < 0 || c.ks > 8) return false;
    return prefill_dense_fits(c);
}

// Time model of the dense form (microseconds, fitted to GB300 timings of
// this kernel over BN x ring depth x K split on the Llama-3.1-8B layers at
// M = 128 and 1920, median error 3 %): a 64-k step costs 0.376 + 0.00069 BN
// (nearly the same for any tile width: each MMA costs about the same at any
// N), plus 3.84 per wave for start-up and epilogue and 1.3 + 0.034 BN for
// the cluster reduction when K is split.  (The fit also has 5.6 per launch.)
static double prefill_dense_cost(int bn, int ks, long long tiles, int K, const DeviceInfo &dev) {
    const int resident = dev.prefill_clusters[ks];
    if (resident <= 0) return 1e30;
    const long long waves = (tiles + resident - 1) / resident;
    const int nwt = (K + kWK - 1) / kWK;
    const int steps = ((nwt + ks - 1) / ks) * kStepsPerW;
    return (double)waves * (steps * (0.376 + 0.00069 * bn) + 3.84 + (ks > 1 ? 1.3 + 0.034 * bn : 0.0));
}

int prefill_dense_best_ks(const PrefillCfg &base, long long tiles, int K, const DeviceInfo &dev, double *cost) {
    const int nwt = (K + kWK - 1) / kWK;
    int best = 1;
    double best_cost = 1e30;
    for (int ks = 1; ks <= 8 && ks <= nwt; ++ks) {
        PrefillCfg c = base;
        c.ks = ks;
        if (!prefill_dense_fits(c)) continue;
        const double t = prefill_dense_cost(c.BN, ks, tiles, K, dev);
        if (t < best_cost * 0.995) {
            best_cost = t;
            best = ks;
        }
    }
    if (cost) *cost = best_cost;
    return best;
}

// The deepest x and A rings (equal depth, at most 4) that fit with c.ks.
static bool prefill_dense_fit_stages(PrefillCfg &c) {
    for (int st = 4; st >= 2; --st) {
        c.stages = c.astages = st;
        if (prefill_dense_fits(c)) return true;
    }
    return false;
}

PrefillCfg prefill_dense_pick_cfg(int M, int N, int K, const DeviceInfo &dev) {
    const int ntiles_n = (N + kBW - 1) / kBW;
    const int bn_max = std::min(256, std::max(16, (M + 15) / 16 * 16));
    PrefillCfg best{bn_max, 2, 2, 0, 1};
    double best_cost = 1e30;
    for (int bn = 16; bn <= bn_max; bn += 16) {
        PrefillCfg c{bn, 2, 2, 0, 1};
        if (!prefill_dense_fit_stages(c)) continue;
        const long long tiles = (long long)((M + bn - 1) / bn) * ntiles_n;
        double t = 0.0;
        // the split needs room for the partial tile over the rings
        PrefillCfg cs = c;
        cs.ks = 2;
        const bool can_split = prefill_dense_fit_stages(cs);
        c.ks = can_split ? prefill_dense_best_ks(cs, tiles, K, dev, &t) : 1;
        if (!can_split) t = prefill_dense_cost(bn, 1, tiles, K, dev);
        if (t < best_cost * 0.995) {
            best_cost = t;
            best = c;
        }
    }
    prefill_dense_fit_stages(best);
    return best;
}

bool prefill_cfg_valid(const PrefillCfg &c) {
    if (c.BN < 16 || c.BN > 256 || c.BN % 16 != 0) return false;
    if (c.swap != 0 && (c.swap != 1 || c.BN != kHalf)) return false;
    if (c.stages < 2 || c.astages < 2 || c.wstages < 2) return false;
    if (c.ks < 0 || c.ks > 8) return false;
    if (c.ks > 1 && !prefill_split_fits(c)) return false;
    return prefill_cfg_fits(c);
}

template <int DT, bool ASYM, bool DENSE>
static cudaError_t launch_t(const CUtensorMap &tx, const CUtensorMap &tw, const CUtensorMap &to,
                            const PrefillParams &p, size_t smem, int grid, cudaStream_t s, bool pdl) {
    auto kern = prefill_kernel<DT, ASYM, DENSE>;
    cudaError_t e = raise_smem_cap(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (p.KS > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = p.KS;
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
    return cudaLaunchKernelEx(&cfg, kern, tx, tw, to, p);
}

// How many clusters of KS CTAs (KS = 1 .. 8) of the prefill kernel the GPU
// holds at once, at the largest shared-memory size (every configuration
// takes more than half an SM's shared memory, so one CTA per SM).
cudaError_t prefill_prepare_device(DeviceInfo &dev) {
    const int smem = dev.max_smem_optin;
    decltype(&prefill_kernel<0, false, false>) kerns[6] = {
        prefill_kernel<0, false, false>, prefill_kernel<0, true, false>, prefill_kernel<1, false, false>,
        prefill_kernel<1, true, false>, prefill_kernel<0, false, true>, prefill_kernel<1, false, true>};
    for (auto k : kerns) {
        const cudaError_t e = raise_smem_cap(reinterpret_cast<const void *>(k), (size_t)smem);
        if (e != cudaSuccess) return e;
    }
    dev.prefill_clusters[0] = 0;
    for (int ks = 1; ks <= 8; ++ks) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ks * 64, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = ks;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kerns[0], &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = ks == 1 ? dev.sm_count : 0;
        }
        dev.prefill_clusters[ks] = n;
    }
    return cudaSuccess;
}

cudaError_t launch_prefill(const GemmArgs &a, const PrefillCfg &c, const DeviceInfo &dev,
                           cudaStream_t s, bool pdl) {
    if (dev.encode_tiled == nullptr) return cudaErrorNotSupported;
    const bool dense = a.wdense != nullptr;
    if (dense ? !prefill_dense_cfg_valid(c) : !prefill_cfg_valid(c)) return cudaErrorInvalidValue;
    EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(dev.encode_tiled);
    const CUtensorMapDataType act = a.dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tx, tw, to;
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)c.BN};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tx, act, 2, const_cast<void *>(a.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (dense) {
        // W [N, K] in the activation dtype: 64-k x 128-row boxes, 128-byte swizzle
        cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.N};
        cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kHalf};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tw, act, 2, const_cast<void *>(a.wdense), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        cuuint64_t dims[2] = {(cuuint64_t)(a.K / 8), (cuuint64_t)a.N};
        cuuint64_t strides[1] = {(cuuint64_t)(a.K / 8) * 4};
        cuuint32_t box[2] = {(cuuint32_t)(kWK / 8), (cuuint32_t)kBW};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t *>(a.qweight), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int ldo = a.ldo > 0 ? a.ldo : a.N;
    {
        // plain: one [BN][256] box; swapped: [BN][64] boxes, 128-byte swizzle
        cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.M};
        cuuint64_t strides[1] = {(cuuint64_t)ldo * 2};
        cuuint32_t box[2] = {(cuuint32_t)(c.swap ? 64 : kBW), (cuuint32_t)c.BN};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&to, act, 2, a.out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   c.swap ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    PrefillParams p;
    p.dq = dq_consts_seq(a.dtype);
    p.scales = (const uint16_t *)a.scales;
    p.qz = a.qzeros;
    p.out = (uint16_t *)a.out;
    p.bias = (const uint16_t *)a.bias;
    p.M = a.M;
    p.N = a.N;
    p.ldo = ldo;
    p.swap = c.swap ? 1 : 0;
    p.K = a.K;
    p.G = dense ? 0 : a.G;
    p.ng = dense ? 0 : a.K / a.G;
    p.BN = c.BN;
    p.SX = c.stages;
    p.SA = c.astages;
    p.SW = dense ? 0 : c.wstages;
    p.n_mtiles = (a.M + c.BN - 1) / c.BN;
    p.status = dev.status;
    const int n_ntiles = (a.N + kBW - 1) / kBW;
    const SmemLayout L = prefill_layout(c.BN, c.stages, c.astages, dense ? 0 : c.wstages);
    // Too few output tiles to fill the SMs (small M): split K over a cluster
    // of KS CTAs, each summing whole packed-weight tiles, as long as every
    // CTA keeps at least one tile and the fp32 partial tile fits over the rings.
    const int tiles = n_ntiles * p.n_mtiles;
    const int nwt = (a.K + kWK - 1) / kWK;
    int ks = c.ks;
    if (ks == 0) ks = dense ? prefill_dense_best_ks(c, tiles, a.K, dev, nullptr) : prefill_best_ks(c, tiles, nwt, dev, nullptr);
    ks = std::max(1, std::min(ks, nwt));
    p.KS = ks;
    const int grid = tiles * ks;
    const size_t smem = L.total;
    const bool asym = a.qzeros != nullptr;
    if (dense)
        return a.dtype == 0 ? launch_t<0, false, true>(tx, tw, to, p, smem, grid, s, pdl)
                            : launch_t<1, false, true>(tx, tw, to, p, smem, grid, s, pdl);
    if (a.dtype == 0)
        return asym ? launch_t<0, true, false>(tx, tw, to, p, smem, grid, s, pdl)
                    : launch_t<0, false, false>(tx, tw, to, p, smem, grid, s, pdl);
    return asym ? launch_t<1, true, false>(tx, tw, to, p, smem, grid, s, pdl)
                : launch_t<1, false, false>(tx, tw, to, p, smem, grid, s, pdl);
}

}  // namespace w4a16
