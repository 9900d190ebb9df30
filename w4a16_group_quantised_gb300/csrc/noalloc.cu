// noalloc.cu -- w4a16_gemm_decode_noalloc: the decode GEMM (M <= 8) on the
// balanced kernel of decode_sk.cu, with its scratch in static device memory,
// so that no call ever allocates.
//
// Who needs it: a caller that must not allocate device memory after start-up
// -- an engine that reserves its whole device arena up front and accounts
// for every byte, or code in a section where a cudaMalloc would synchronise
// the device or is not allowed at all.  w4a16_gemm itself allocates once per
// device (the balanced kernel's workspace, on its first call); this entry
// point never does.
//
// Scratch: a file-scope workspace of partial-sum slots (two slots of
// [16 rows][8 m] fp32 per CTA, one CTA per SM, up to kMaxSMs SMs) and one
// ticket counter per 16-row block (up to kMaxRowBlocks, i.e. N <= 131072).
// Larger problems or devices are rejected with W4A16_ERR_SHAPE /
// W4A16_ERR_DEVICE, and so is a K whose staged x (M x K) and partial slots
// do not fit in the kernel's shared memory (decode_sk_applicable, for
// example M = 8 with K = 14336).  Every device has its own copy of these
// arrays; the first call on a device, with that device current, looks up
// their addresses (cudaGetSymbolAddress) and clears the counters, so that
// first call should come before any stream capture: made during a capture
// it returns W4A16_ERR_DEVICE without touching the device, and a later call
// outside the capture sets up as usual.  A set-up that fails is retried by
// the next call.  The kernel returns every counter to zero itself.
//
// Programmatic dependent launch follows the library's switch (W4A16_PDL,
// w4a16_debug_set_config(3)) as w4a16_gemm does.
//
// All calls on one device share the scratch: calls whose kernels overlap on
// the GPU (for instance on two streams without an ordering between them)
// race on it and give wrong results.  Calls issued in order on one stream
// are safe (the kernel touches the scratch only after its grid-dependency
// wait).
#include <mutex>

#include "kernels.h"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kMaxSMs = 256;
constexpr int kSlotFloats = 2 * 128;                 // per CTA: two [16][8] fp32 partial slots
constexpr int kMaxRowBlocks = 8192;                  // 16-row blocks: N <= 131072

static __device__ __align__(256) float g_noalloc_ws[kMaxSMs * kSlotFloats];       // 256 KB
static __device__ __align__(256) int g_noalloc_counters[kMaxRowBlocks];           // 32 KB

constexpr int kMaxDevices = 64;
struct NoAllocState {
    std::mutex mu;
    bool ready = false;
    int rc = W4A16_ERR_DEVICE;
    DeviceInfo info{};
    float *ws = nullptr;
    int *counters = nullptr;
};
NoAllocState g_state[kMaxDevices];

// Sets st.rc; st.ready only on success (a failed set-up is retried by the next call).
void set_up(NoAllocState &st, int dev) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.info.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    if (major != 10 || minor != 3 || st.info.sm_count > kMaxSMs) {
        st.rc = W4A16_ERR_DEVICE;
        return;
    }
    void *ws = nullptr, *counters = nullptr;
    if (cudaGetSymbolAddress(&ws, g_noalloc_ws) != cudaSuccess ||
        cudaGetSymbolAddress(&counters, g_noalloc_counters) != cudaSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    st.info.status = device_status_word();
    if (st.info.status == nullptr ||
        cudaMemset(counters, 0, sizeof(int) * kMaxRowBlocks) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    st.info.device = dev;
    st.ws = static_cast<float *>(ws);
    st.counters = static_cast<int *>(counters);
    st.rc = W4A16_OK;
    st.ready = true;
}

}  // namespace
}  // namespace w4a16

extern "C" int w4a16_gemm_decode_noalloc(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                                         const int32_t *qzeros_or_null, int G, int N, void *out,
                                         w4a16_stream_t stream, w4a16_dtype_t dtype) {
    using namespace w4a16;
    int rc = validate_gemm_args(x, M, K, qweight, scales, qzeros_or_null, G, N, out, (int)dtype);
    if (rc != W4A16_OK) return rc;
    if (M > W4A16_MAX_DECODE_M) return W4A16_ERR_SHAPE;
    if ((N + 15) / 16 > kMaxRowBlocks || !decode_sk_applicable(M, K)) return W4A16_ERR_SHAPE;
    if (M == 0) return W4A16_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_DEVICE;
    NoAllocState &st = g_state[dev];
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    {
        std::lock_guard<std::mutex> lk(st.mu);
        if (!st.ready) {
            // set-up synchronises the device: never during a capture
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return W4A16_ERR_CUDA;
            if (cs != cudaStreamCaptureStatusNone) return W4A16_ERR_DEVICE;
            set_up(st, dev);
            if (!st.ready) return st.rc;
        }
    }
    GemmArgs a{x, qweight, scales, qzeros_or_null, out, M, N, K, G, (int)dtype};
    const cudaError_t e = launch_decode_sk(a, 4, st.info, st.ws, st.counters, s, pdl_for_stream(s));
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}
