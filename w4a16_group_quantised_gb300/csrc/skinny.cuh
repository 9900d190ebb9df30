// skinny.cuh -- the multiply step shared by the skinny-M decode kernels.
//
// A lane holds one packed word (8 weights, k .. k+7) of weight rows g and
// g+8 of a 16-row block; dq_word_i4 turns each into four (k, k+4) pairs and
// two m16n8k16 MMAs (weights = A, x = B, fp32 accumulate) consume them.  The
// two MMAs of a word go to different accumulators, and consecutive words of a
// lane may alternate between two such pairs, so two or four independent
// accumulation chains keep the tensor pipe's result latency off the critical
// path.  The asm statements are not volatile: they have no side effects
// beyond their outputs, and the compiler may interleave them with the loads
// of the next words.
#pragma once
#include "dequant.cuh"

namespace w4a16 {

template <int DT>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
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

// One word of rows g (wa) and g+8 (wb): 16 weights, two MMAs into c0 and c1.
// xv = the matching x pairs: (x_k, x_k+4), (x_k+1, x_k+5), (x_k+2, x_k+6),
// (x_k+3, x_k+7) of batch column g.
template <int DT>
__device__ __forceinline__ void mac_word(float (&c0)[4], float (&c1)[4], const DqConsts &dc, uint32_t wa, uint32_t wb,
                                         uint32_t zla, uint32_t zha, uint32_t s2a, uint32_t zlb, uint32_t zhb,
                                         uint32_t s2b, uint4 xv) {
    uint32_t oa[4], ob[4];
    dq_word_i4_rt<DT>(wa, dc, zla, zha, s2a, oa);
    dq_word_i4_rt<DT>(wb, dc, zlb, zhb, s2b, ob);
    mma16816<DT>(c0, oa[0], ob[0], oa[1], ob[1], xv.x, xv.y);
    mma16816<DT>(c1, oa[2], ob[2], oa[3], ob[3], xv.z, xv.w);
}

// Four words of rows g and g+8 (one 128-k block row chunk) into NC = 4
// chains (words alternate between the pairs (0, 1) and (2, 3)) or NC = 2
// chains (every word into (0, 1)).
template <int DT, int NC>
__device__ __forceinline__ void mac_block(float (&acc)[NC][4], const DqConsts &dc, uint4 wa, uint4 wb, uint32_t zla,
                                          uint32_t zha, uint32_t s2a, uint32_t zlb, uint32_t zhb, uint32_t s2b,
                                          const uint4 (&xv)[4]) {
    constexpr int P = NC == 4 ? 2 : 0;
    mac_word<DT>(acc[0], acc[1], dc, wa.x, wb.x, zla, zha, s2a, zlb, zhb, s2b, xv[0]);
    mac_word<DT>(acc[P], acc[P + 1], dc, wa.y, wb.y, zla, zha, s2a, zlb, zhb, s2b, xv[1]);
    mac_word<DT>(acc[0], acc[1], dc, wa.z, wb.z, zla, zha, s2a, zlb, zhb, s2b, xv[2]);
    mac_word<DT>(acc[P], acc[P + 1], dc, wa.w, wb.w, zla, zha, s2a, zlb, zhb, s2b, xv[3]);
}

// Sum of the chains, element e, in a fixed order.
template <int NC>
__device__ __forceinline__ float chain_sum(const float (&acc)[NC][4], int e) {
    if (NC == 4) return (acc[0][e] + acc[1][e]) + (acc[2 % NC][e] + acc[3 % NC][e]);
    return acc[0][e] + acc[1][e];
}

// zhi2 from zlo2 (see dequant.cuh).
template <int DT>
__device__ __forceinline__ uint32_t zhi_from_zlo(uint32_t zl2) {
    return zhi_from_zlo_dq<DT>(zl2);
}

template <int DT>
__device__ __forceinline__ uint16_t f32_to_dt(float v) {
    if (DT == 0) {
        __half h = __float2half_rn(v);
        return *reinterpret_cast<uint16_t *>(&h);
    }
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t *>(&h);
}

template <int DT>
__device__ __forceinline__ float dt_to_f32(uint16_t v) {
    if (DT == 0) return __half2float(__ushort_as_half(v));
    return __bfloat162float(__ushort_as_bfloat16(v));
}

// Plain C++ loads from the dynamic shared-memory block (the compiler
// schedules them freely between the barrier waits, which carry memory
// clobbers).  The kernels derive their aligned base by pointer arithmetic on
// the __shared__ array itself, so the compiler keeps the shared address
// space and emits shared-memory loads and stores, not generic ones (a
// uintptr_t round trip loses it: the prefill kernel's dequantisers measured
// 4-5 % slower that way).
__device__ __forceinline__ uint4 sh_v4(const unsigned char *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ uint2 sh_v2(const unsigned char *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint32_t sh_u32(const unsigned char *p) { return *reinterpret_cast<const uint32_t *>(p); }

}  // namespace w4a16
