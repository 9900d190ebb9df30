// dequant.cuh -- int4 -> fp16/bf16 dequantisation in registers (sm_103a).
//
// The weight is w = RN_dtype((q - z) * s).  "[ROCm][Kernel] Add
// HybridW4A16LinearKernel: Triton prefill + HIP skinny decode", PR
// description, names the idea for bf16 (a magic-number dequant that avoids a
// round trip through fp32); the constants below follow from the IEEE-754
// layouts alone:
//
//   * OR-ing a 4-bit value n into the low fraction bits of a float whose
//     fraction is zero and whose unit in the last place (ulp) is 1 gives
//     exactly M + n (M = 1024 = 0x6400 in fp16, M = 128 = 0x4300 in bf16).
//   * If the nibble sits 4 bits higher (bits 4..7 of a 16-bit lane), a
//     magic whose ulp is 1/16 does the same: fp16 0x5400 = 64.0 has ulp
//     64 / 2^10 = 1/16.  bf16 has only 7 fraction bits, so there the nibble
//     is moved to bits 3..6 and the magic is 0x4180 = 16.0 (ulp 1/8).
//   * (M + q) - (M + z) = q - z is exact (a small integer), and one RN
//     multiply by s then rounds the exact product (q - z) * s once -- the same
//     value as the definition, bit for bit.  The subtraction and the multiply
//     are kept as two operations on purpose: folding them into one fused
//     multiply-add would round the constant (M + z) * s first.
//
// Two pairings of the eight nibbles of a word are provided:
//   dq_word_seq : registers hold (k, k+1) pairs in natural order -- for
//                 operands written to shared memory (prefill, debug output);
//   dq_word_i4  : registers hold (k, k+4) pairs -- cheaper (no byte
//                 permutes); the decode kernel feeds its x operand in the
//                 matching order, so the dot product is unchanged.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace w4a16 {

template <int DT> struct Dtype;
template <> struct Dtype<0> {
    using T = __half;
    using T2 = __half2;
    static constexpr uint32_t kMagicLo = 0x6400;  // 1024.0, ulp 1
    static constexpr uint32_t kMagicHi = 0x5400;  // 64.0, ulp 1/16 (nibble at bits 4..7)
};
template <> struct Dtype<1> {
    using T = __nv_bfloat16;
    using T2 = __nv_bfloat162;
    static constexpr uint32_t kMagicLo = 0x4300;  // 128.0, ulp 1
    static constexpr uint32_t kMagicHi = 0x4180;  // 16.0, ulp 1/8 (nibble at bits 3..6)
};

__device__ __forceinline__ uint32_t rep2(uint32_t h) { return h | (h << 16); }

// Packed 2 x 16-bit subtract / multiply on raw 32-bit registers, each one
// IEEE operation rounded to nearest even (no contraction into an FMA).
template <int DT>
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    uint32_t r;
    if (DT == 0)
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

template <int DT>
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t r;
    if (DT == 0)
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Subtrahend (M + z) for the "low" magic, in both lanes.
template <int DT>
__device__ __forceinline__ uint32_t zlo2(uint32_t z) { return rep2(Dtype<DT>::kMagicLo | z); }

// Subtrahend (M' + z) for the "high" magic, in both lanes: fp16 64 + z has z
// in fraction bits 4..7; bf16 16 + z has z in fraction bits 3..6.
template <int DT>
__device__ __forceinline__ uint32_t zhi2(uint32_t z) {
    return rep2(Dtype<DT>::kMagicHi | (DT == 0 ? (z << 4) : (z << 3)));
}

// The masks and magic words of the two pairings, held in registers.  The
// kernels take them from their launch parameters, so the compiler cannot
// turn them back into immediates: a three-input logic operation accepts at
// most one immediate, and (x & mask) | magic with two immediates costs two
// instructions instead of one.
struct DqConsts {
    uint32_t m0, m1;   // nibble masks
    uint32_t g0, g1;   // magic words (both lanes)
};

// (k, k+4) pairing (dq_word_i4_rt): fp16 nibbles at bits 0..3 / 4..7 of each
// lane; bf16 nibbles at bits 0..3 / 3..6.
__host__ __device__ inline DqConsts dq_consts_i4(int dtype) {
    if (dtype == 0) return DqConsts{0x000F000Fu, 0x00F000F0u, 0x64006400u, 0x54005400u};
    return DqConsts{0x000F000Fu, 0x00780078u, 0x43004300u, 0x41804180u};
}
// natural pairing (dq_word_seq_rt): fp16 low lane bits 0..3 (magic 1024),
// high lane bits 4..7 (magic 64); bf16 both lanes bits 0..3 (magic 128).
__host__ __device__ inline DqConsts dq_consts_seq(int dtype) {
    if (dtype == 0) return DqConsts{0x00F0000Fu, 0u, 0x54006400u, 0u};
    return DqConsts{0x000F000Fu, 0u, 0x43004300u, 0u};
}

template <int DT>
__device__ __forceinline__ void dq_word_i4_rt(uint32_t w, const DqConsts &c, uint32_t zl2, uint32_t zh2,
                                              uint32_t s2, uint32_t (&o)[4]) {
    uint32_t v0, v1, v2, v3;
    const uint32_t w8 = w >> 8;
    v0 = (w & c.m0) | c.g0;
    v2 = (w8 & c.m0) | c.g0;
    if (DT == 0) {
        v1 = (w & c.m1) | c.g1;
        v3 = (w8 & c.m1) | c.g1;
    } else {
        v1 = ((w >> 1) & c.m1) | c.g1;
        v3 = ((w >> 9) & c.m1) | c.g1;
    }
    o[0] = hmul2_u<DT>(hsub2_u<DT>(v0, zl2), s2);
    o[1] = hmul2_u<DT>(hsub2_u<DT>(v1, zh2), s2);
    o[2] = hmul2_u<DT>(hsub2_u<DT>(v2, zl2), s2);
    o[3] = hmul2_u<DT>(hsub2_u<DT>(v3, zh2), s2);
}

template <int DT>
__device__ __forceinline__ void dq_word_seq_rt(uint32_t w, const DqConsts &c, uint32_t zc2, uint32_t s2,
                                               uint32_t (&o)[4]) {
    if (DT == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t b = __byte_perm(w, 0u, (uint32_t)(i | (i << 8)));
            o[i] = hmul2_u<0>(hsub2_u<0>((b & c.m0) | c.g0, zc2), s2);
        }
    } else {
        const uint32_t t = w >> 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t b = __byte_perm(w, t, (uint32_t)(i | ((4 + i) << 8)));
            o[i] = hmul2_u<1>(hsub2_u<1>((b & c.m0) | c.g0, zc2), s2);
        }
    }
}

// Natural-order pairs.  o[i] = (w_{2i}, w_{2i+1}) for nibbles 2i, 2i+1 of word.
// zc2 = (M_lo + z, M_hi + z) for fp16, (M_lo + z, M_lo + z) for bf16; s2 = (s, s).
template <int DT>
__device__ __forceinline__ uint32_t zseq2(uint32_t z) {
    if (DT == 0) return (Dtype<0>::kMagicLo | z) | ((Dtype<0>::kMagicHi | (z << 4)) << 16);
    return rep2(Dtype<1>::kMagicLo | z);
}

template <int DT>
__device__ __forceinline__ void dq_word_seq(uint32_t w, uint32_t zc2, uint32_t s2, uint32_t (&o)[4]) {
    if (DT == 0) {
        // byte i -> both halves; low lane keeps bits 0..3 (n_2i, magic 1024),
        // high lane keeps bits 4..7 (n_2i+1, magic 64 with ulp 1/16).
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t b = __byte_perm(w, 0u, (uint32_t)(i | (i << 8)));
            uint32_t v = (b & 0x00F0000Fu) | 0x54006400u;
            o[i] = hmul2_u<0>(hsub2_u<0>(v, zc2), s2);
        }
    } else {
        uint32_t t = w >> 4;  // byte i of t has nibble 2i+1 in its low half
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t b = __byte_perm(w, t, (uint32_t)(i | ((4 + i) << 8)));
            uint32_t v = (b & 0x000F000Fu) | 0x43004300u;
            o[i] = hmul2_u<1>(hsub2_u<1>(v, zc2), s2);
        }
    }
}

// (k, k+4) pairs.  o[0] = (w0, w4), o[1] = (w1, w5), o[2] = (w2, w6), o[3] = (w3, w7).
// zl2 = zlo2(z), zh2 = zhi2(z); s2 = (s, s).
template <int DT>
__device__ __forceinline__ void dq_word_i4(uint32_t w, uint32_t zl2, uint32_t zh2, uint32_t s2,
                                           uint32_t (&o)[4]) {
    uint32_t v0, v1, v2, v3;
    if (DT == 0) {
        uint32_t w8 = w >> 8;
        v0 = (w & 0x000F000Fu) | 0x64006400u;    // nibbles 0, 4   -> 1024 + n
        v1 = (w & 0x00F000F0u) | 0x54005400u;    // nibbles 1, 5   -> 64 + n
        v2 = (w8 & 0x000F000Fu) | 0x64006400u;   // nibbles 2, 6
        v3 = (w8 & 0x00F000F0u) | 0x54005400u;   // nibbles 3, 7
    } else {
        v0 = (w & 0x000F000Fu) | 0x43004300u;            // nibbles 0, 4 -> 128 + n
        v1 = ((w >> 1) & 0x00780078u) | 0x41804180u;     // nibbles 1, 5 -> 16 + n
        v2 = ((w >> 8) & 0x000F000Fu) | 0x43004300u;     // nibbles 2, 6
        v3 = ((w >> 9) & 0x00780078u) | 0x41804180u;     // nibbles 3, 7
    }
    o[0] = hmul2_u<DT>(hsub2_u<DT>(v0, zl2), s2);
    o[1] = hmul2_u<DT>(hsub2_u<DT>(v1, zh2), s2);
    o[2] = hmul2_u<DT>(hsub2_u<DT>(v2, zl2), s2);
    o[3] = hmul2_u<DT>(hsub2_u<DT>(v3, zh2), s2);
}

// zhi2 from zlo2: the same zero point moved from the low-magic to the
// high-magic position in both lanes (as the decode kernels derive it).
template <int DT>
__device__ __forceinline__ uint32_t zhi_from_zlo_dq(uint32_t zl2) {
    return ((zl2 & 0x000F000Fu) << (DT == 0 ? 4 : 3)) | rep2(Dtype<DT>::kMagicHi);
}

// Zero point of row n, group g: nibble n%8 of qzeros[n/8, g]; 8 when symmetric.
__device__ __forceinline__ uint32_t zero_point(const int32_t *qz, int n, int g, int ng) {
    if (qz == nullptr) return 8u;
    return ((uint32_t)__ldg(qz + (size_t)(n >> 3) * ng + g) >> (4 * (n & 7))) & 0xFu;
}

}  // namespace w4a16
