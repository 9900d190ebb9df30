// api.cu -- the C ABI of include/w4a16.h: argument validation, per-device
// state, the M dispatcher and the end-to-end host-buffer form.
//
// The dispatcher follows "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton
// prefill + HIP skinny decode", PR description: small batch sizes (the page
// uses M <= 5) go to the skinny split-K decode kernel, larger ones to the
// fused-dequant GEMM.  Here the threshold (decode_max_m, used by
// select_path_impl) is the measured crossover between the two kernels, which
// on GB300 is the decode kernel's own limit, M <= 8.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>

#include "w4a16.h"
#include "kernels.h"

// Device status word: kernels whose bounded waits run out write here.
__device__ int g_w4a16_status;

namespace w4a16 {
namespace {

constexpr int kMaxDevices = 64;

// Balanced-decode-kernel scratch of one stream: CTA partial slots and
// per-row-block tickets (zero between calls).  Calls on one stream run in
// order, so they never share it concurrently.
struct StreamScratch {
    cudaStream_t stream;
    float *ws;
    int *cnt;
};
constexpr int kMaxStreamScratch = 64;

struct DevState {
    std::once_flag once;
    int rc = W4A16_ERR_DEVICE;
    DeviceInfo info{};
    std::mutex scratch_mu;
    int n_scratch = 0;
    StreamScratch scratch[kMaxStreamScratch];
};
DevState g_dev[kMaxDevices];

// Tuning overrides (process-wide), set through w4a16_debug_set_config.
std::mutex g_cfg_mu;
bool g_decode_override = false;
DecodeCfg g_decode_cfg{};
bool g_prefill_override = false;
PrefillCfg g_prefill_cfg{};
int g_prefill_split = 0;   // > 0: every prefill call splits its weight rows there (test hook)
int g_pdl = 1;
// Kernel-selection log to stderr (environment W4A16_LOG): 0 off, 1 each
// distinct selection once, 2 every call.
int g_log = 0;
std::mutex g_log_mu;
uint64_t g_log_seen[512];
int g_n_log_seen = 0;

void log_selection(const char *line) {
    int mode;
    {
        std::lock_guard<std::mutex> lk(g_cfg_mu);
        mode = g_log;
    }
    if (mode <= 0) return;
    std::lock_guard<std::mutex> lk(g_log_mu);
    if (mode == 1) {
        uint64_t h = 1469598103934665603ull;              // FNV-1a of the line
        for (const char *c = line; *c; ++c) h = (h ^ (unsigned char)*c) * 1099511628211ull;
        for (int i = 0; i < g_n_log_seen; ++i)
            if (g_log_seen[i] == h) return;
        if (g_n_log_seen < 512) g_log_seen[g_n_log_seen++] = h;
    }
    std::fprintf(stderr, "w4a16: %s\n", line);
}
// balanced decode kernel: enabled flag and preferred ring depth
int g_sk_on = 0, g_sk_ns = 4;
// test hook (w4a16_debug_set_config(7)): decode kernels issue no weight copies
int g_hold_copies = 0;
// Streams whose last library launch wrote weights (w4a16_pack,
// w4a16_pack_zeros): the next GEMM on such a stream is launched without
// programmatic dependent launch, because the GEMM kernels read weights
// before their grid-dependency wait.
std::mutex g_pdl_mu;
cudaStream_t g_pdl_unsafe[16];
int g_n_pdl_unsafe = 0;

void mark_weights_written(cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_pdl_mu);
    for (int i = 0; i < g_n_pdl_unsafe; ++i)
        if (g_pdl_unsafe[i] == s) return;
    if (g_n_pdl_unsafe < 16) g_pdl_unsafe[g_n_pdl_unsafe++] = s;
    else g_pdl_unsafe[15] = s;
}

// true (and the mark cleared) if the last library launch on s wrote weights
bool take_weights_written(cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_pdl_mu);
    for (int i = 0; i < g_n_pdl_unsafe; ++i)
        if (g_pdl_unsafe[i] == s) {
            g_pdl_unsafe[i] = g_pdl_unsafe[--g_n_pdl_unsafe];
            return true;
        }
    return false;
}

void init_device(DevState &st, int dev) {
    DeviceInfo &d = st.info;
    d.device = dev;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    if (major != 10 || minor != 3) {  // the kernels are built for sm_103a only
        st.rc = W4A16_ERR_DEVICE;
        return;
    }
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    void *sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_w4a16_status) != cudaSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    d.status = static_cast<int *>(sym);
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    d.encode_tiled = fn;
    if (prefill_prepare_device(d) != cudaSuccess) {
        st.rc = W4A16_ERR_CUDA;
        return;
    }
    const char *e = std::getenv("W4A16_PDL");
    const char *lg = std::getenv("W4A16_LOG");
    {
        std::lock_guard<std::mutex> lk(g_cfg_mu);
        if (e && e[0] == '0') g_pdl = 0;
        if (lg) g_log = std::atoi(lg);
    }
    st.rc = W4A16_OK;
}

int get_device(const DeviceInfo **out, DevState **state = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_DEVICE;
    DevState &st = g_dev[dev];
    std::call_once(st.once, init_device, std::ref(st), dev);
    if (st.rc != W4A16_OK) return st.rc;
    *out = &st.info;
    if (state) *state = &st;
    return W4A16_OK;
}

// The balanced decode kernel's scratch for stream s, made on the first call
// that enables that kernel on s (one cudaMalloc of the partial slots and one
// of the tickets, which are cleared on s).  Returns false, allocating
// nothing, while s is being captured or when the table is full; the caller
// then uses the cluster kernel, which needs no scratch.  The default path
// never gets here, so a default w4a16_gemm call never allocates.
bool stream_scratch(DevState &st, cudaStream_t s, float **ws, int **cnt) {
    std::lock_guard<std::mutex> lk(st.scratch_mu);
    for (int i = 0; i < st.n_scratch; ++i)
        if (st.scratch[i].stream == s) {
            *ws = st.scratch[i].ws;
            *cnt = st.scratch[i].cnt;
            return true;
        }
    if (st.n_scratch == kMaxStreamScratch) return false;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return false;
    }
    const size_t wsf = decode_sk_workspace_floats(st.info.sm_count);
    float *w = nullptr;
    int *c = nullptr;
    if (cudaMalloc(&w, wsf * sizeof(float)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (cudaMalloc(&c, sizeof(int) * kDecodeTickets) != cudaSuccess ||
        cudaMemsetAsync(c, 0, sizeof(int) * kDecodeTickets, s) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(w);
        if (c) cudaFree(c);
        return false;
    }
    st.scratch[st.n_scratch++] = StreamScratch{s, w, c};
    *ws = w;
    *cnt = c;
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_common(int M, int N, int K, int G, int dtype) {
    if (dtype != W4A16_F16 && dtype != W4A16_BF16) return W4A16_ERR_DTYPE;
    if (G != 32 && G != 64 && G != 128) return W4A16_ERR_GROUP;
    if (M < 0 || N <= 0 || K <= 0) return W4A16_ERR_SHAPE;
    if (K % G != 0) return W4A16_ERR_GROUP;
    if (N % 8 != 0) return W4A16_ERR_SHAPE;
    // int32 index headroom for the kernels' per-row arithmetic
    if ((long long)N * (K / 8) >= (1LL << 31) || (long long)M * K >= (1LL << 31) ||
        (long long)M * N >= (1LL << 31))
        return W4A16_ERR_SHAPE;
    return W4A16_OK;
}

int validate_gemm(const void *x, int M, int K, const int32_t *qw, const void *scales,
                  const int32_t *qz, int G, int N, const void *out, int dtype) {
    int rc = validate_common(M, N, K, G, dtype);
    if (rc != W4A16_OK) return rc;
    if (qw == nullptr || scales == nullptr) return W4A16_ERR_NULL;
    if (M > 0 && (x == nullptr || out == nullptr)) return W4A16_ERR_NULL;
    if (!aligned16(qw) || !aligned16(scales) || !aligned16(qz) || !aligned16(x) || !aligned16(out))
        return W4A16_ERR_ALIGN;
    return W4A16_OK;
}

// Largest M the decode kernel takes for this problem.  Measured on GB300
// (bench.py --crossover: 2560x9728, 19456x2560 and 4096x14336, G = 32, 64,
// 128, symmetric and asymmetric, fp16 and bf16, L2 flushed before every
// launch): the decode kernel is the faster one at every M it supports (the
// prefill kernel takes 1.6x to 9.7x as long at M <= 8), so the threshold is
// the decode kernel's own limit in every cell.  The pages route M <= 5 to
// their skinny kernel ("[ROCm][Kernel] Add HybridW4A16LinearKernel", PR
// description).
int decode_max_m(int N, int K, int G, int sym, int dtype) {
    (void)N; (void)K; (void)G; (void)sym; (void)dtype;
    return W4A16_MAX_DECODE_M;
}

int select_path_impl(int M, int N, int K, int G, int sym, int dtype) {
    return M <= decode_max_m(N, K, G, sym, dtype) ? W4A16_PATH_DECODE : W4A16_PATH_PREFILL;
}

// A prefill plan: one launch, or the two row blocks of a split -- rows
// [0, n_split) in whole waves of wide tiles, then the rest, each writing its
// columns of y.
static cudaError_t launch_prefill_plan(const GemmArgs &a, const PrefillPlan &plan, const DeviceInfo &dev,
                                       cudaStream_t s, bool pdl) {
    if (plan.n_split >= a.N) return launch_prefill(a, plan.main, dev, s, pdl);
    cudaError_t e = launch_prefill(prefill_rows(a, 0, plan.n_split), plan.main, dev, s, pdl);
    if (e == cudaSuccess) e = launch_prefill(prefill_rows(a, plan.n_split, a.N - plan.n_split), plan.tail, dev, s, pdl);
    return e;
}

int run_gemm(const void *x, int M, int K, const int32_t *qw, const void *scales, const int32_t *qz,
             int G, int N, void *out, w4a16_stream_t stream, int dtype, int path,
             const void *bias = nullptr, int epilogue = W4A16_EPI_NONE) {
    int rc = validate_gemm(x, M, K, qw, scales, qz, G, N, out, dtype);
    if (rc != W4A16_OK) return rc;
    if (path != W4A16_PATH_AUTO && path != W4A16_PATH_DECODE && path != W4A16_PATH_PREFILL)
        return W4A16_ERR_ARG;
    if (epilogue != W4A16_EPI_NONE && epilogue != W4A16_EPI_SILU_MUL) return W4A16_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(bias) & 1u) != 0) return W4A16_ERR_ALIGN;
    if (path == W4A16_PATH_DECODE && M > W4A16_MAX_DECODE_M) return W4A16_ERR_SHAPE;
    if (epilogue == W4A16_EPI_SILU_MUL) {
        if (path == W4A16_PATH_PREFILL) return W4A16_ERR_ARG;
        if (M > W4A16_MAX_DECODE_M) return W4A16_ERR_SHAPE;
        path = W4A16_PATH_DECODE;
    }
    if (M == 0) return W4A16_OK;
    const DeviceInfo *dev = nullptr;
    DevState *st = nullptr;
    rc = get_device(&dev, &st);
    if (rc != W4A16_OK) return rc;
    if (path == W4A16_PATH_AUTO) path = select_path_impl(M, N, K, G, qz == nullptr, dtype);

    GemmArgs a{x, qw, scales, qz, out, M, N, K, G, dtype};
    a.bias = bias;
    a.silu_mul = epilogue == W4A16_EPI_SILU_MUL ? 1 : 0;
    const bool plain = bias == nullptr && epilogue == W4A16_EPI_NONE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool asym = qz != nullptr;
    bool pdl;
    {
        std::lock_guard<std::mutex> lk(g_cfg_mu);
        pdl = g_pdl != 0;
    }
    if (take_weights_written(s)) pdl = false;
    cudaError_t e;
    if (path == W4A16_PATH_DECODE) {
        int sk_on, ns_pref;
        bool cluster_override, hold;
        DecodeCfg c;
        {
            std::lock_guard<std::mutex> lk(g_cfg_mu);
            hold = g_hold_copies != 0;
            sk_on = g_sk_on && !g_decode_override;
            ns_pref = g_sk_ns;
            cluster_override = g_decode_override;
            c = g_decode_cfg;
        }
        float *ws = nullptr;
        int *cnt = nullptr;
        if (plain && !hold && sk_on && (N + 15) / 16 <= kDecodeTickets && decode_sk_applicable(M, K) &&
            stream_scratch(*st, s, &ws, &cnt)) {
            e = launch_decode_sk(a, ns_pref, *dev, ws, cnt, s, pdl);
            char line[256];
            std::snprintf(line, sizeof line, "gemm M=%d N=%d K=%d G=%d %s %s path=decode kernel=decode_sk ring=%d pdl=%d",
                          M, N, K, G, dtype == 0 ? "fp16" : "bf16", asym ? "asym" : "sym", ns_pref, pdl ? 1 : 0);
            log_selection(line);
            return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
        }
        if (!cluster_override)
            c = decode_pick_cfg(M, N, K, G, qz == nullptr, dtype, dev->sm_count, dev->smem_per_sm);
        if (!decode_cfg_valid(c, M, K, G, asym)) return W4A16_ERR_ARG;
        e = launch_decode(a, c, *dev, s, pdl, hold);
        {
            const int RT = 16 * c.R * c.NW;
            const int tiles = a.silu_mul ? (N / 2 + RT / 2 - 1) / (RT / 2) : (N + RT - 1) / RT;
            char line[320];
            std::snprintf(line, sizeof line,
                          "gemm M=%d N=%d K=%d G=%d %s %s path=decode kernel=decode_kernel R=%d NW=%d NB=%d NS=%d "
                          "S=%d grid=%d pdl=%d bias=%d epilogue=%s%s",
                          M, N, K, G, dtype == 0 ? "fp16" : "bf16", asym ? "asym" : "sym", c.R, c.NW, c.NB, c.NS,
                          c.S, tiles * c.S, pdl ? 1 : 0, bias != nullptr ? 1 : 0,
                          a.silu_mul ? "silu_mul" : "none", cluster_override ? " (forced)" : "");
            log_selection(line);
        }
    } else {
        PrefillPlan plan;
        bool forced;
        int split_at;
        {
            std::lock_guard<std::mutex> lk(g_cfg_mu);
            forced = g_prefill_override;
            split_at = g_prefill_split;
            plan.main = plan.tail = g_prefill_cfg;
            plan.n_split = N;
        }
        if (!forced) plan = prefill_pick_plan(M, N, K, false, *dev);
        else if (!prefill_cfg_valid(plan.main)) return W4A16_ERR_ARG;   // fits the dense form only
        if (!forced && split_at > 0 && split_at < N) {   // test hook: a split where asked, each part picked
            plan.n_split = split_at;
            plan.main = prefill_pick_cfg(M, split_at, K, G, qz == nullptr, dtype, *dev);
            plan.tail = prefill_pick_cfg(M, N - split_at, K, G, qz == nullptr, dtype, *dev);
        }
        e = launch_prefill_plan(a, plan, *dev, s, pdl);
        char line[400];
        const PrefillCfg &c = plan.main, &t = plan.tail;
        if (plan.n_split >= N)
            std::snprintf(line, sizeof line,
                          "gemm M=%d N=%d K=%d G=%d %s %s path=prefill kernel=prefill_kernel BN=%d x_stages=%d "
                          "a_stages=%d w_stages=%d ks=%d swap=%d pdl=%d bias=%d%s",
                          M, N, K, G, dtype == 0 ? "fp16" : "bf16", asym ? "asym" : "sym", c.BN, c.stages,
                          c.astages, c.wstages, c.ks, c.swap, pdl ? 1 : 0, bias != nullptr ? 1 : 0,
                          forced ? " (forced)" : "");
        else
            std::snprintf(line, sizeof line,
                          "gemm M=%d N=%d K=%d G=%d %s %s path=prefill kernel=prefill_kernel rows 0..%d: BN=%d "
                          "x_stages=%d a_stages=%d w_stages=%d ks=%d swap=%d; rows %d..%d: BN=%d x_stages=%d "
                          "a_stages=%d w_stages=%d ks=%d swap=%d; pdl=%d bias=%d",
                          M, N, K, G, dtype == 0 ? "fp16" : "bf16", asym ? "asym" : "sym", plan.n_split, c.BN,
                          c.stages, c.astages, c.wstages, c.ks, c.swap, plan.n_split, N, t.BN, t.stages, t.astages,
                          t.wstages, t.ks, t.swap, pdl ? 1 : 0, bias != nullptr ? 1 : 0);
        log_selection(line);
    }
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

// Dense-weight GEMM (the dequantised prefill cache) on the prefill kernel.
int run_gemm_dense(const void *x, int M, int K, const void *w, int N, const void *bias, void *out, int dtype,
                   w4a16_stream_t stream) {
    if (dtype != W4A16_F16 && dtype != W4A16_BF16) return W4A16_ERR_DTYPE;
    if (M < 0 || N <= 0 || K <= 0 || N % 8 != 0 || K % 8 != 0) return W4A16_ERR_SHAPE;
    if ((long long)M * K >= (1LL << 31) || (long long)N * K >= (1LL << 31) || (long long)M * N >= (1LL << 31))
        return W4A16_ERR_SHAPE;
    if (w == nullptr) return W4A16_ERR_NULL;
    if (M > 0 && (x == nullptr || out == nullptr)) return W4A16_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out)) return W4A16_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(bias) & 1u) != 0) return W4A16_ERR_ALIGN;
    if (M == 0) return W4A16_OK;
    const DeviceInfo *dev = nullptr;
    int rc = get_device(&dev);
    if (rc != W4A16_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bool pdl;
    bool forced;
    int split_at;
    PrefillPlan plan;
    {
        std::lock_guard<std::mutex> lk(g_cfg_mu);
        pdl = g_pdl != 0;
        forced = g_prefill_override;
        split_at = g_prefill_split;
        plan.main = plan.tail = g_prefill_cfg;
        plan.n_split = N;
    }
    if (take_weights_written(s)) pdl = false;
    if (!forced) plan = prefill_pick_plan(M, N, K, true, *dev);
    if (!forced && split_at > 0 && split_at < N) {   // test hook: a split where asked, each part picked
        plan.n_split = split_at;
        plan.main = prefill_dense_pick_cfg(M, split_at, K, *dev);
        plan.tail = prefill_dense_pick_cfg(M, N - split_at, K, *dev);
    }
    plan.main.wstages = plan.tail.wstages = 0;
    if (!prefill_dense_cfg_valid(plan.main) || !prefill_dense_cfg_valid(plan.tail)) return W4A16_ERR_ARG;
    GemmArgs a{x, nullptr, nullptr, nullptr, out, M, N, K, 0, dtype};
    a.bias = bias;
    a.wdense = w;
    const cudaError_t e = launch_prefill_plan(a, plan, *dev, s, pdl);
    const PrefillCfg &c = plan.main, &t = plan.tail;
    char line[320];
    if (plan.n_split >= N)
        std::snprintf(line, sizeof line,
                      "gemm_dense M=%d N=%d K=%d %s path=prefill kernel=prefill_kernel(dense) BN=%d stages=%d ks=%d "
                      "pdl=%d bias=%d%s",
                      M, N, K, dtype == 0 ? "fp16" : "bf16", c.BN, c.stages, c.ks, pdl ? 1 : 0,
                      bias != nullptr ? 1 : 0, forced ? " (forced)" : "");
    else
        std::snprintf(line, sizeof line,
                      "gemm_dense M=%d N=%d K=%d %s path=prefill kernel=prefill_kernel(dense) rows 0..%d: BN=%d "
                      "stages=%d ks=%d; rows %d..%d: BN=%d stages=%d ks=%d; pdl=%d bias=%d",
                      M, N, K, dtype == 0 ? "fp16" : "bf16", plan.n_split, c.BN, c.stages, c.ks, plan.n_split, N,
                      t.BN, t.stages, t.ks, pdl ? 1 : 0, bias != nullptr ? 1 : 0);
    log_selection(line);
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

}  // namespace

cudaError_t raise_smem_cap(const void *func, size_t need) {
    struct Entry {
        const void *func;
        int device;
    };
    static std::mutex mu;
    static Entry done[256];
    static int n_done = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].func == func && done[i].device == dev) return cudaSuccess;   // already at the maximum
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    if (need > (size_t)optin) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    if (n_done < 256) done[n_done++] = Entry{func, dev};
    return cudaSuccess;
}

// Shared with the allocation-free entry point (noalloc.cu): the same host
// validation, and the status word's device address (no device state is
// created here).
int validate_gemm_args(const void *x, int M, int K, const int32_t *qw, const void *scales, const int32_t *qz,
                       int G, int N, const void *out, int dtype) {
    return validate_gemm(x, M, K, qw, scales, qz, G, N, out, dtype);
}

bool pdl_enabled() {
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    return g_pdl != 0;
}

bool pdl_for_stream(cudaStream_t s) {
    const bool on = pdl_enabled();
    return take_weights_written(s) ? false : on;
}

int *device_status_word() {
    void *sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_w4a16_status) != cudaSuccess) return nullptr;
    return static_cast<int *>(sym);
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

int w4a16_pack(const uint8_t *q, int N, int K, int32_t *qweight, w4a16_stream_t stream) {
    if (N < 0 || K < 0 || K % 8 != 0) return W4A16_ERR_SHAPE;
    if ((long long)N * K >= (1LL << 34)) return W4A16_ERR_SHAPE;
    if (N == 0 || K == 0) return W4A16_OK;
    if (q == nullptr || qweight == nullptr) return W4A16_ERR_NULL;
    if (!aligned16(q) || !aligned16(qweight)) return W4A16_ERR_ALIGN;
    const DeviceInfo *dev = nullptr;
    int rc = get_device(&dev);
    if (rc != W4A16_OK) return rc;
    if (launch_pack(q, N, K, qweight, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return W4A16_ERR_CUDA;
    mark_weights_written(reinterpret_cast<cudaStream_t>(stream));
    return W4A16_OK;
}

int w4a16_pack_zeros(const uint8_t *z, int N, int n_groups, int32_t *qzeros, w4a16_stream_t stream) {
    if (N < 0 || n_groups < 0 || N % 8 != 0) return W4A16_ERR_SHAPE;
    if ((long long)N * n_groups >= (1LL << 31)) return W4A16_ERR_SHAPE;
    if (N == 0 || n_groups == 0) return W4A16_OK;
    if (z == nullptr || qzeros == nullptr) return W4A16_ERR_NULL;
    if (!aligned16(z) || !aligned16(qzeros)) return W4A16_ERR_ALIGN;
    const DeviceInfo *dev = nullptr;
    int rc = get_device(&dev);
    if (rc != W4A16_OK) return rc;
    if (launch_pack_zeros(z, N, n_groups, qzeros, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4A16_ERR_CUDA;
    mark_weights_written(reinterpret_cast<cudaStream_t>(stream));
    return W4A16_OK;
}

int w4a16_dequant_debug_ex(const int32_t *qweight, const void *scales, const int32_t *qzeros_or_null, int G,
                           int N, int K, void *out, w4a16_dtype_t dtype, w4a16_stream_t stream, int routine) {
    if (routine < W4A16_DQ_PREFILL || routine > W4A16_DQ_BALANCED) return W4A16_ERR_ARG;
    int rc = validate_common(0, N, K, G, (int)dtype);
    if (rc != W4A16_OK) return rc;
    if (qweight == nullptr || scales == nullptr || out == nullptr) return W4A16_ERR_NULL;
    if (!aligned16(qweight) || !aligned16(scales) || !aligned16(qzeros_or_null) || !aligned16(out))
        return W4A16_ERR_ALIGN;
    const DeviceInfo *dev = nullptr;
    rc = get_device(&dev);
    if (rc != W4A16_OK) return rc;
    return launch_dequant(qweight, scales, qzeros_or_null, G, N, K, out, (int)dtype, routine,
                          reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? W4A16_OK
               : W4A16_ERR_CUDA;
}

int w4a16_dequant_debug(const int32_t *qweight, const void *scales, const int32_t *qzeros_or_null,
                        int G, int N, int K, void *out, w4a16_dtype_t dtype, w4a16_stream_t stream) {
    return w4a16_dequant_debug_ex(qweight, scales, qzeros_or_null, G, N, K, out, dtype, stream, W4A16_DQ_PREFILL);
}

int w4a16_gemm(const void *x, int M, int K, const int32_t *qweight, const void *scales,
               const int32_t *qzeros_or_null, int G, int N, void *out, w4a16_stream_t stream,
               w4a16_dtype_t dtype) {
    return run_gemm(x, M, K, qweight, scales, qzeros_or_null, G, N, out, stream, (int)dtype,
                    W4A16_PATH_AUTO);
}

int w4a16_gemm_f16(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                   const int32_t *qzeros_or_null, int G, int N, void *out, w4a16_stream_t stream) {
    return run_gemm(x, M, K, qweight, scales, qzeros_or_null, G, N, out, stream, W4A16_F16,
                    W4A16_PATH_AUTO);
}

int w4a16_gemm_bf16(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                    const int32_t *qzeros_or_null, int G, int N, void *out, w4a16_stream_t stream) {
    return run_gemm(x, M, K, qweight, scales, qzeros_or_null, G, N, out, stream, W4A16_BF16,
                    W4A16_PATH_AUTO);
}

int w4a16_gemm_ex(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                  const int32_t *qzeros_or_null, int G, int N, void *out, w4a16_stream_t stream,
                  w4a16_dtype_t dtype, w4a16_path_t path) {
    return run_gemm(x, M, K, qweight, scales, qzeros_or_null, G, N, out, stream, (int)dtype, (int)path);
}

int w4a16_gemm_fused(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                     const int32_t *qzeros_or_null, int G, int N, const void *bias_or_null, int epilogue,
                     void *out, w4a16_stream_t stream, w4a16_dtype_t dtype, w4a16_path_t path) {
    return run_gemm(x, M, K, qweight, scales, qzeros_or_null, G, N, out, stream, (int)dtype, (int)path,
                    bias_or_null, epilogue);
}

int w4a16_moe_gemm(const void *x, int T, int K, const int32_t *qweight, const void *scales,
                   const int32_t *qzeros_or_null, int G, int N, int E, const int32_t *expert_ids, int topk,
                   const float *route_weights_or_null, void *out, w4a16_dtype_t dtype, w4a16_stream_t stream) {
    if (T < 0 || E < 1 || topk < 1) return W4A16_ERR_SHAPE;
    int rc = validate_common(1, N, K, G, (int)dtype);
    if (rc != W4A16_OK) return rc;
    const long long slots = (long long)T * topk;
    if ((long long)E * N * (K / 8) >= (1LL << 31) || (long long)E * N >= (1LL << 31) ||
        slots * N >= (1LL << 31) || (long long)T * K >= (1LL << 31) || slots > (1LL << 24))
        return W4A16_ERR_SHAPE;
    if (qweight == nullptr || scales == nullptr) return W4A16_ERR_NULL;
    if (T > 0 && (x == nullptr || out == nullptr || expert_ids == nullptr)) return W4A16_ERR_NULL;
    if (!aligned16(qweight) || !aligned16(scales) || !aligned16(qzeros_or_null) || !aligned16(x) ||
        !aligned16(out) || (reinterpret_cast<uintptr_t>(expert_ids) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(route_weights_or_null) & 3u) != 0)
        return W4A16_ERR_ALIGN;
    if (T == 0) return W4A16_OK;
    const DeviceInfo *dev = nullptr;
    rc = get_device(&dev);
    if (rc != W4A16_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bool pdl, forced;
    DecodeCfg c;
    {
        std::lock_guard<std::mutex> lk(g_cfg_mu);
        pdl = g_pdl != 0;
        forced = g_decode_override;
        c = g_decode_cfg;
    }
    if (take_weights_written(s)) pdl = false;
    const bool asym = qzeros_or_null != nullptr;
    if (!forced) c = decode_pick_cfg(1, N, K, G, !asym, (int)dtype, dev->sm_count, dev->smem_per_sm, (int)slots);
    if (!decode_cfg_valid(c, 1, K, G, asym)) return W4A16_ERR_ARG;
    GemmArgs a{x, qweight, scales, qzeros_or_null, out, 1, N, K, G, (int)dtype};
    a.expert_ids = expert_ids;
    a.route_w = route_weights_or_null;
    a.n_experts = E;
    a.topk = topk;
    a.n_slots = (int)slots;
    const cudaError_t e = launch_decode(a, c, *dev, s, pdl);
    char line[320];
    std::snprintf(line, sizeof line,
                  "moe_gemm T=%d topk=%d E=%d N=%d K=%d G=%d %s %s path=decode kernel=decode_kernel(experts) R=%d "
                  "NW=%d NB=%d NS=%d S=%d pdl=%d%s",
                  T, topk, E, N, K, G, dtype == 0 ? "fp16" : "bf16", asym ? "asym" : "sym", c.R, c.NW, c.NB, c.NS,
                  c.S, pdl ? 1 : 0, forced ? " (forced)" : "");
    log_selection(line);
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_dequantize(const int32_t *qweight, const void *scales, const int32_t *qzeros_or_null, int G, int N,
                     int K, void *w_out, w4a16_dtype_t dtype, w4a16_stream_t stream) {
    return w4a16_dequant_debug_ex(qweight, scales, qzeros_or_null, G, N, K, w_out, dtype, stream, W4A16_DQ_PREFILL);
}


int w4a16_gemm_dense(const void *x, int M, int K, const void *w, int N, const void *bias_or_null, void *out,
                     w4a16_dtype_t dtype, w4a16_stream_t stream) {
    return run_gemm_dense(x, M, K, w, N, bias_or_null, out, (int)dtype, stream);
}

int w4a16_gemm_cached(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                      const int32_t *qzeros_or_null, int G, int N, const void *w_cache_or_null, void *out,
                      w4a16_stream_t stream, w4a16_dtype_t dtype) {
    int rc = validate_gemm(x, M, K, qweight, scales, qzeros_or_null, G, N, out, (int)dtype);
    if (rc != W4A16_OK) return rc;
    if (w_cache_or_null != nullptr &&
        select_path_impl(M, N, K, G, qzeros_or_null == nullptr, (int)dtype) == W4A16_PATH_PREFILL)
        return run_gemm_dense(x, M, K, w_cache_or_null, N, nullptr, out, (int)dtype, stream);
    return run_gemm(x, M, K, qweight, scales, qzeros_or_null, G, N, out, stream, (int)dtype, W4A16_PATH_AUTO);
}

int w4a16_gemm_chain(const void *x, int M, const w4a16_layer_t *layers, int n_layers, w4a16_dtype_t dtype,
                     w4a16_stream_t stream) {
    if (n_layers < 0) return W4A16_ERR_ARG;
    if (n_layers > 0 && layers == nullptr) return W4A16_ERR_NULL;
    // validate the whole chain before enqueuing anything
    const void *in = x;
    for (int i = 0; i < n_layers; ++i) {
        const w4a16_layer_t &L = layers[i];
        int rc = validate_gemm(in, M, L.K, L.qweight, L.scales, L.qzeros_or_null, L.G, L.N, L.out, (int)dtype);
        if (rc != W4A16_OK) return rc;
        if (L.epilogue != W4A16_EPI_NONE && L.epilogue != W4A16_EPI_SILU_MUL) return W4A16_ERR_ARG;
        if ((reinterpret_cast<uintptr_t>(L.bias_or_null) & 1u) != 0) return W4A16_ERR_ALIGN;
        if (L.epilogue == W4A16_EPI_SILU_MUL && M > W4A16_MAX_DECODE_M) return W4A16_ERR_SHAPE;
        if (i > 0) {
            const w4a16_layer_t &P = layers[i - 1];
            const int width = P.epilogue == W4A16_EPI_SILU_MUL ? P.N / 2 : P.N;
            if (L.K != width) return W4A16_ERR_SHAPE;
        }
        in = L.out;
    }
    in = x;
    for (int i = 0; i < n_layers; ++i) {
        const w4a16_layer_t &L = layers[i];
        int rc = run_gemm(in, M, L.K, L.qweight, L.scales, L.qzeros_or_null, L.G, L.N, L.out, stream, (int)dtype,
                          W4A16_PATH_AUTO, L.bias_or_null, L.epilogue);
        if (rc != W4A16_OK) return rc;
        in = L.out;
    }
    return W4A16_OK;
}

int w4a16_gemm_host_async(const void *x_host, int M, int K, const int32_t *qweight, const void *scales,
                          const int32_t *qzeros_or_null, int G, int N, void *out_host, w4a16_dtype_t dtype,
                          void *x_dev, void *out_dev, w4a16_stream_t stream) {
    int rc = validate_gemm(x_dev, M, K, qweight, scales, qzeros_or_null, G, N, out_dev, (int)dtype);
    if (rc != W4A16_OK) return rc;
    if (M > 0 && (x_host == nullptr || out_host == nullptr)) return W4A16_ERR_NULL;
    if (M == 0) return W4A16_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(x_dev, x_host, (size_t)M * K * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return W4A16_ERR_CUDA;
    rc = run_gemm(x_dev, M, K, qweight, scales, qzeros_or_null, G, N, out_dev, stream, (int)dtype,
                  W4A16_PATH_AUTO);
    if (rc != W4A16_OK) return rc;
    if (cudaMemcpyAsync(out_host, out_dev, (size_t)M * N * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return W4A16_ERR_CUDA;
    return W4A16_OK;
}

int w4a16_gemm_host(const void *x_host, int M, int K, const int32_t *qweight, const void *scales,
                    const int32_t *qzeros_or_null, int G, int N, void *out_host, w4a16_dtype_t dtype,
                    void *x_dev, void *out_dev, w4a16_stream_t stream) {
    int rc = w4a16_gemm_host_async(x_host, M, K, qweight, scales, qzeros_or_null, G, N, out_host, dtype, x_dev,
                                   out_dev, stream);
    if (rc != W4A16_OK || M == 0) return rc;
    return cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A16_OK
                                                                                         : W4A16_ERR_CUDA;
}

int w4a16_select_path(int M, int N, int K, int G, int sym, int dtype) {
    int rc = validate_common(M, N, K, G, dtype);
    if (rc != W4A16_OK) return rc;
    return select_path_impl(M, N, K, G, sym != 0, dtype);
}

int w4a16_debug_decode_trace(unsigned long long *trace_buf, const int *nk) {
    const DeviceInfo *dev = nullptr;
    int rc = get_device(&dev);
    if (rc != W4A16_OK) return rc;
    if (trace_buf != nullptr && (nk == nullptr || (reinterpret_cast<uintptr_t>(trace_buf) & 7u) != 0))
        return W4A16_ERR_ARG;
    // cudaErrorNotSupported: a buffer given to a library built without the trace
    return decode_trace_install(trace_buf, trace_buf != nullptr ? nk : nullptr) == cudaSuccess ? W4A16_OK
                                                                                               : W4A16_ERR_ARG;
}

int w4a16_debug_prefill_plan(int M, int N, int K, int dense, int sm_count, const int *clusters, int *out) {
    if (M <= 0 || N <= 0 || K <= 0 || N % 8 != 0 || K % 8 != 0 || sm_count <= 0 || clusters == nullptr ||
        out == nullptr)
        return W4A16_ERR_ARG;
    DeviceInfo dev{};
    dev.sm_count = sm_count;
    dev.prefill_clusters[0] = 0;
    for (int k = 1; k <= 8; ++k) {
        if (clusters[k - 1] < 0) return W4A16_ERR_ARG;
        dev.prefill_clusters[k] = clusters[k - 1];
    }
    const PrefillPlan plan = prefill_pick_plan(M, N, K, dense != 0, dev);
    const PrefillCfg *cs[2] = {&plan.main, &plan.tail};
    out[0] = plan.n_split;
    for (int i = 0; i < 2; ++i) {
        out[1 + 6 * i] = cs[i]->BN;
        out[2 + 6 * i] = cs[i]->stages;
        out[3 + 6 * i] = cs[i]->astages;
        out[4 + 6 * i] = cs[i]->wstages;
        out[5 + 6 * i] = cs[i]->ks;
        out[6 + 6 * i] = cs[i]->swap;
    }
    return W4A16_OK;
}

int w4a16_last_device_error(void) {
    const DeviceInfo *dev = nullptr;
    int rc = get_device(&dev);
    if (rc != W4A16_OK) return rc;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_w4a16_status, sizeof(int)) != cudaSuccess) return W4A16_ERR_CUDA;
    return v;
}

int w4a16_clear_device_error(void) {
    const DeviceInfo *dev = nullptr;
    DevState *st = nullptr;
    int rc = get_device(&dev, &st);
    if (rc != W4A16_OK) return rc;
    int z = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return W4A16_ERR_CUDA;
    // A kernel that gave up a wait may have left tickets counted: clear them.
    {
        std::lock_guard<std::mutex> lk(st->scratch_mu);
        for (int i = 0; i < st->n_scratch; ++i)
            if (cudaMemset(st->scratch[i].cnt, 0, sizeof(int) * kDecodeTickets) != cudaSuccess) return W4A16_ERR_CUDA;
    }
    if (cudaMemcpyToSymbol(g_w4a16_status, &z, sizeof(int)) != cudaSuccess) return W4A16_ERR_CUDA;
    return cudaDeviceSynchronize() == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_version(void) { return 100; }

// Tuning hook: which = 1 sets the decode configuration {R, NW, NB, NS, S},
// which = 2 the prefill configuration {BN, x stages, A stages, W stages};
// n = 0 clears it.
// which = 3 sets programmatic dependent launch on (vals[0] != 0) or off.
int w4a16_debug_set_config(int which, const int *vals, int n) {
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    if (which == 1) {
        if (n == 0) { g_decode_override = false; return W4A16_OK; }
        if (n != 5 || vals == nullptr) return W4A16_ERR_ARG;
        g_decode_cfg = DecodeCfg{vals[0], vals[1], vals[2], vals[3], vals[4]};
        g_decode_override = true;
        return W4A16_OK;
    }
    if (which == 2) {
        if (n == 0) { g_prefill_override = false; return W4A16_OK; }
        if ((n < 4 || n > 6) || vals == nullptr) return W4A16_ERR_ARG;
        PrefillCfg c{vals[0], vals[1], vals[2], vals[3], n >= 5 ? vals[4] : 0};
        c.swap = n == 6 ? vals[5] : 0;
        PrefillCfg cd = c;              // the dense form has no packed-weight ring
        cd.wstages = 0;
        if (!prefill_cfg_valid(c) && !prefill_dense_cfg_valid(cd)) return W4A16_ERR_ARG;
        g_prefill_cfg = c;
        g_prefill_override = true;
        return W4A16_OK;
    }
    if (which == 3) {
        if (n != 1 || vals == nullptr) return W4A16_ERR_ARG;
        g_pdl = vals[0] != 0;
        return W4A16_OK;
    }
    if (which == 8) {
        if (n == 0) { g_prefill_split = 0; return W4A16_OK; }
        if (n != 1 || vals == nullptr || vals[0] <= 0 || vals[0] % 256 != 0) return W4A16_ERR_ARG;
        g_prefill_split = vals[0];
        return W4A16_OK;
    }
    if (which == 7) {
        if (n == 0) { g_hold_copies = 0; return W4A16_OK; }
        if (n != 1 || vals == nullptr) return W4A16_ERR_ARG;
        g_hold_copies = vals[0] != 0;
        return W4A16_OK;
    }
    if (which == 4) {
        if (n == 0) { g_sk_on = 0; g_sk_ns = 4; return W4A16_OK; }
        if (n != 2 || vals == nullptr) return W4A16_ERR_ARG;
        if (vals[0] < 0 || vals[0] > 1 || (vals[1] != 2 && vals[1] != 4 && vals[1] != 6))
            return W4A16_ERR_ARG;
        g_sk_on = vals[0];
        g_sk_ns = vals[1];
        return W4A16_OK;
    }
    return W4A16_ERR_ARG;
}

}  // extern "C"
