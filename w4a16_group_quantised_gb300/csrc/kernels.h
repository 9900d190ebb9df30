// kernels.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; the public interface is include/w4a16.h.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

struct GemmArgs {
    const void *x;
    const int32_t *qweight;
    const void *scales;
    const int32_t *qzeros;  // nullptr: symmetric
    void *out;
    int M, N, K, G;
    int dtype;              // 0 fp16, 1 bf16
    const void *bias = nullptr;  // [N] in the activation dtype, or none
    const void *wdense = nullptr;  // prefill only: dtype W [N, K] (dequantised cache) instead of qweight
    // decode expert mode (MoE): qweight/scales/qzeros stack n_experts experts of N rows;
    // x [T, K], out [n_slots = T * topk, N], expert_ids / route_w [n_slots] on the device
    const int *expert_ids = nullptr;
    const float *route_w = nullptr;
    int n_experts = 0, topk = 0, n_slots = 0;
    int silu_mul = 0;       // 1: out [M, N/2] = silu(y[:, :N/2]) * y[:, N/2:] (rows 0..N/2-1 = gate)
    int ldo = 0;            // prefill only: elements between output rows (0: N)
};

// Per-device facts the launchers need.
struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
    int smem_per_sm;        // shared memory of one SM (all resident CTAs together)
    int *status;            // device address of the status word
    void *encode_tiled;     // cuTensorMapEncodeTiled entry point
    int prefill_clusters[9];  // prefill kernel: clusters of k CTAs resident at once (k = 1..8)
};

// ---- pack.cu
cudaError_t launch_pack(const uint8_t *q, int N, int K, int32_t *qweight, cudaStream_t s);
cudaError_t launch_pack_zeros(const uint8_t *z, int N, int ng, int32_t *qzeros, cudaStream_t s);
cudaError_t launch_dequant(const int32_t *qweight, const void *scales, const int32_t *qzeros,
                           int G, int N, int K, void *out, int dtype, int routine, cudaStream_t s);

// ---- decode.cu
struct DecodeCfg {
    int R;    // 16-row blocks per warp (1, 2)
    int NW;   // warps per CTA (1, 2, 4, 8); a CTA owns 16 * R * NW rows
    int NB;   // TMA boxes (128 k each) per ring stage (1..8)
    int NS;   // ring stages (2..8)
    int S;    // CTAs along K in a cluster (1..8)
};
// slots > 1: an MoE launch of `slots` expert matrices of N rows each (one token each)
DecodeCfg decode_pick_cfg(int M, int N, int K, int G, int sym, int dtype, int sm_count, int smem_per_sm,
                          int slots = 1);
// Decode timeline hook: buf (device, kTraceLayers x kTraceCtas x kTraceEvents
// uint64) or null to turn it off; nk = (N, K) of up to four traced layers.
// Only the trace build (W4A16_DECODE_TRACE) records anything; the default
// build returns cudaErrorNotSupported for a non-null buf.
constexpr int kTraceLayers = 4, kTraceCtas = 512, kTraceEvents = 8;
cudaError_t decode_trace_install(unsigned long long *buf, const int *nk);
bool decode_cfg_valid(const DecodeCfg &c, int M, int K, int G, bool asym);
size_t decode_smem_bytes(const DecodeCfg &c, int M, int K, int G, bool asym);
// hold_copies: test hook -- the kernel issues no weight copies, so its bounded
// waits run out and it exits with W4A16_ERR_TIMEOUT in the status word.
cudaError_t launch_decode(const GemmArgs &a, const DecodeCfg &c, const DeviceInfo &dev,
                          cudaStream_t s, bool pdl, bool hold_copies = false);

// Per-stream scratch of the balanced decode kernel: kDecodeTickets ints
// (zero between calls) and decode_sk_workspace_floats(sm_count) floats.
constexpr int kDecodeTickets = 1 << 16;

// ---- decode_sk.cu (balanced skinny kernel; needs a per-device workspace)
size_t decode_sk_smem_bytes(int M, int K);
size_t decode_sk_workspace_floats(int sm_count);
bool decode_sk_applicable(int M, int K);
cudaError_t launch_decode_sk(const GemmArgs &a, int ns, const DeviceInfo &dev, float *ws, int *counters,
                             cudaStream_t s, bool pdl);

// Make sure kernel `func` may launch with `need` bytes of dynamic shared
// memory on the current device.  The cap is a property of the function,
// shared by every launch of it and read again whenever a captured graph node
// of it is launched on its own (as a profiler does), so it is set once to
// the device's opt-in maximum and never lowered: setting it per launch let a
// smaller launch lower it under a graph node captured with a larger one.
cudaError_t raise_smem_cap(const void *func, size_t need);

// ---- api.cu helpers used by noalloc.cu
int validate_gemm_args(const void *x, int M, int K, const int32_t *qw, const void *scales, const int32_t *qz,
                       int G, int N, const void *out, int dtype);
int *device_status_word();
// Whether the next GEMM on s may use programmatic dependent launch: the
// process-wide switch (W4A16_PDL, w4a16_debug_set_config(3)), and not right
// after a library launch on s that wrote weights.  Clears that mark.
bool pdl_for_stream(cudaStream_t s);

// ---- prefill.cu
struct PrefillCfg {
    int BN;       // tokens per tile (MMA N), multiple of 16, <= 256
    int stages;   // x-tile ring stages (64 k each)
    int astages;  // dequantised-weight ring stages
    int wstages;  // packed-weight ring stages (256 k each)
    int ks = 0;   // CTAs of a cluster splitting K: 0 = chosen at launch, else 1..8
    int swap = 0; // 1: x is the MMA's A operand and the 256 weight rows B (BN must be 128)
};
bool prefill_cfg_valid(const PrefillCfg &c);
// dense form (wdense): no packed-weight ring (wstages unused)
bool prefill_dense_cfg_valid(const PrefillCfg &c);
PrefillCfg prefill_dense_pick_cfg(int M, int N, int K, const DeviceInfo &dev);
int prefill_dense_best_ks(const PrefillCfg &base, long long tiles, int K, const DeviceInfo &dev, double *cost);
PrefillCfg prefill_pick_cfg(int M, int N, int K, int G, int sym, int dtype, const DeviceInfo &dev);
// The fused path's launch plan: weight rows [0, n_split) with `main`, and,
// when n_split < N, rows [n_split, N) as a second launch with `tail`.
struct PrefillPlan {
    PrefillCfg main;
    int n_split;
    PrefillCfg tail;
};
PrefillPlan prefill_pick_plan(int M, int N, int K, bool dense, const DeviceInfo &dev);
// The part of a prefill problem on weight rows [n0, n0 + rows): offset operands, same x and output rows.
GemmArgs prefill_rows(const GemmArgs &a, int n0, int rows);
cudaError_t launch_prefill(const GemmArgs &a, const PrefillCfg &c, const DeviceInfo &dev,
                           cudaStream_t s, bool pdl);
cudaError_t prefill_prepare_device(DeviceInfo &dev);

}  // namespace w4a16
