// pack.cu -- packing of 4-bit weights and zero points, and the debug
// dequantisation kernel (materialises RN_dtype((q - z) * s) with the
// register routine of a chosen GEMM kernel).
//
// Formats: "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP
// skinny decode", PR description (weights [N, K//8], 8 per int32 along K);
// "Upstream sync 67/N: merge 382bbd5144 HybridW4A16LinearKernel (conflict)",
// section "Upstream's Python side is kept -- and it does NOT work here"
// (zero points int32 [N/8, groups], 8 x uint4 along dim 0).
#include "dequant.cuh"
#include "kernels.h"

namespace w4a16 {

// One thread per output word: q[n, 8j .. 8j+7] -> qweight[n, j].
__global__ void pack_kernel(const uint8_t *__restrict__ q, long long words, int K8,
                            int32_t *__restrict__ qw) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < words;
         i += (long long)gridDim.x * blockDim.x) {
        uint2 b = *reinterpret_cast<const uint2 *>(q + i * 8);  // 8 bytes, 8-aligned
        uint32_t w = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            w |= ((b.x >> (8 * e)) & 0xFu) << (4 * e);
            w |= ((b.y >> (8 * e)) & 0xFu) << (4 * (e + 4));
        }
        qw[i] = (int32_t)w;
    }
    (void)K8;
}

// One thread per output word: z[8r .. 8r+7, g] -> qzeros[r, g].
__global__ void pack_zeros_kernel(const uint8_t *__restrict__ z, int rows8, int ng,
                                  int32_t *__restrict__ qz) {
    long long total = (long long)rows8 * ng;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        int r = (int)(i / ng), g = (int)(i % ng);
        uint32_t w = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) w |= ((uint32_t)z[(size_t)(8 * r + e) * ng + g] & 0xFu) << (4 * e);
        qz[i] = (int32_t)w;
    }
}

// One thread per weight word: 8 outputs (16 bytes) of row n, in natural k
// order, computed by the dequantisation routine a GEMM kernel uses:
//   ROUTINE 0: dq_word_seq_rt with the prefill kernel's constants;
//   ROUTINE 1: dq_word_i4_rt with the cluster decode kernel's constants and
//              its zero-point words (zlo2, and zhi_from_zlo for asymmetric
//              weights / zhi2(8) for symmetric ones), the (k, k+4) pairs put
//              back in natural order;
//   ROUTINE 2: dq_word_i4 (immediate constants), as the balanced decode
//              kernel runs it.
template <int DT, int ROUTINE>
__global__ void dequant_kernel(const int32_t *__restrict__ qw, const uint16_t *__restrict__ scales,
                               const int32_t *__restrict__ qz, int G, int N, int K, DqConsts dc,
                               uint4 *__restrict__ out) {
    const int K8 = K >> 3, ng = K / G;
    long long total = (long long)N * K8;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        int n = (int)(i / K8), j = (int)(i % K8);
        int g = (j * 8) / G;
        uint32_t z = zero_point(qz, n, g, ng);
        uint32_t s = scales[(size_t)n * ng + g];
        uint32_t o[4];
        const uint32_t w = (uint32_t)qw[i];
        if (ROUTINE == 0) {
            dq_word_seq_rt<DT>(w, dc, zseq2<DT>(z), rep2(s), o);
            out[i] = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            const uint32_t zl = zlo2<DT>(z);
            const uint32_t zh = qz != nullptr ? zhi_from_zlo_dq<DT>(zl) : zhi2<DT>(8u);
            if (ROUTINE == 1)
                dq_word_i4_rt<DT>(w, dc, zl, zh, rep2(s), o);
            else
                dq_word_i4<DT>(w, zl, zh, rep2(s), o);
            // o = (w0, w4), (w1, w5), (w2, w6), (w3, w7) -> natural order
            out[i] = make_uint4(__byte_perm(o[0], o[1], 0x5410), __byte_perm(o[2], o[3], 0x5410),
                                __byte_perm(o[0], o[1], 0x7632), __byte_perm(o[2], o[3], 0x7632));
        }
    }
}

static int grid_for(long long work, int threads) {
    long long b = (work + threads - 1) / threads;
    if (b > 152 * 32) b = 152 * 32;
    if (b < 1) b = 1;
    return (int)b;
}

cudaError_t launch_pack(const uint8_t *q, int N, int K, int32_t *qweight, cudaStream_t s) {
    long long words = (long long)N * (K / 8);
    if (words == 0) return cudaSuccess;
    pack_kernel<<<grid_for(words, 256), 256, 0, s>>>(q, words, K / 8, qweight);
    return cudaGetLastError();
}

cudaError_t launch_pack_zeros(const uint8_t *z, int N, int ng, int32_t *qzeros, cudaStream_t s) {
    long long words = (long long)(N / 8) * ng;
    if (words == 0) return cudaSuccess;
    pack_zeros_kernel<<<grid_for(words, 256), 256, 0, s>>>(z, N / 8, ng, qzeros);
    return cudaGetLastError();
}

template <int DT>
static void launch_dequant_t(int routine, int grid, cudaStream_t s, const int32_t *qweight, const uint16_t *scales,
                             const int32_t *qzeros, int G, int N, int K, uint4 *out) {
    if (routine == 0)
        dequant_kernel<DT, 0><<<grid, 256, 0, s>>>(qweight, scales, qzeros, G, N, K, dq_consts_seq(DT), out);
    else if (routine == 1)
        dequant_kernel<DT, 1><<<grid, 256, 0, s>>>(qweight, scales, qzeros, G, N, K, dq_consts_i4(DT), out);
    else
        dequant_kernel<DT, 2><<<grid, 256, 0, s>>>(qweight, scales, qzeros, G, N, K, dq_consts_i4(DT), out);
}

cudaError_t launch_dequant(const int32_t *qweight, const void *scales, const int32_t *qzeros,
                           int G, int N, int K, void *out, int dtype, int routine, cudaStream_t s) {
    long long words = (long long)N * (K / 8);
    if (words == 0) return cudaSuccess;
    int grid = grid_for(words, 256);
    if (dtype == 0)
        launch_dequant_t<0>(routine, grid, s, qweight, (const uint16_t *)scales, qzeros, G, N, K, (uint4 *)out);
    else
        launch_dequant_t<1>(routine, grid, s, qweight, (const uint16_t *)scales, qzeros, G, N, K, (uint4 *)out);
    return cudaGetLastError();
}

}  // namespace w4a16
