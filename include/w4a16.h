/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 group-quantised linear layer.
 *
 *     y[M, N] = x[M, K] . dequant(W)^T,   dequant(W)[n, k] = RN_dtype((q - z) * s)
 *
 * What the operation is comes from "[ROCm][Kernel] Add HybridW4A16LinearKernel:
 * Triton prefill + HIP skinny decode" (vllm-project/vllm#40977), PR
 * description: one weight tensor packed [N, K/8] shared by a skinny decode
 * kernel and a fused-dequant prefill GEMM routed by batch size M; symmetric
 * weights with a fixed bias of 8 (uint4b8) or asymmetric weights with
 * per-group zero points; group sizes 32, 64, 128.  The packed zero-point
 * form comes from "Upstream sync 67/N: merge 382bbd5144
 * HybridW4A16LinearKernel (conflict)" (ROCm/vllm#1175), section "Upstream's
 * Python side is kept -- and it does NOT work here": int32 [N/8, groups],
 * 8 x uint4 along dim 0.
 *
 * Layouts (all row-major, contiguous, on the current CUDA device):
 *   x        fp16/bf16 [M, K]
 *   qweight  int32 [N, K/8]; element k = 8j + i of row n is bits [4i, 4i+3]
 *            of qweight[n, j] (sequential nibble order, fixed by this header)
 *   scales   same dtype as x, [N, K/G]; group g covers k in [gG, (g+1)G)
 *   qzeros   int32 [N/8, K/G] or NULL; z[n, g] is bits [4(n%8), 4(n%8)+3] of
 *            qzeros[n/8, g].  NULL means symmetric: z = 8 for every weight.
 *   out      same dtype as x, [M, N]
 * Arithmetic: the weight is rounded once into the activation dtype (round to
 * nearest even) from the exact product (q - z) * s; the dot products are
 * accumulated in fp32 and rounded once into the output dtype.
 *
 * Ownership: the caller owns every buffer.  Entry points do not allocate,
 * free or synchronise, except: w4a16_gemm_host synchronises its stream to
 * return the host result; w4a16_clear_device_error synchronises the device;
 * the opt-in balanced decode kernel (w4a16_debug_set_config(4)) allocates
 * its per-stream scratch on the first call that uses it on a stream.  Per-device state (SM count, kernel attributes,
 * the tensor-map encoder) is set up on the first call on each device; make
 * that first call outside stream capture.
 *
 * Programmatic dependent launch: the GEMM kernels are launched so that they
 * may start while the kernel before them on the stream is still running,
 * and they read qweight, scales and qzeros before waiting for it (x, out
 * only after).  So the kernel immediately before a GEMM on its stream must
 * not write that GEMM's weights, scales or zero points.  The library's own
 * w4a16_pack / w4a16_pack_zeros are handled: the next GEMM on the same
 * stream is launched without early start.  Anything else that writes
 * weights (a copy, a user kernel) needs some other work or an event between
 * it and the GEMM, or early start switched off (environment W4A16_PDL=0 or
 * w4a16_debug_set_config(3, {0}, 1)).
 *
 * Kernel-selection log: with the environment variable W4A16_LOG=1 (read on
 * the first call on a device) each GEMM entry point prints the kernel it
 * launched -- path, kernel, its configuration, grid, early start, epilogue
 * -- to stderr, each distinct line once; W4A16_LOG=2 prints every call.
 *
 * Errors: arguments are validated on the host before anything is launched;
 * an invalid call returns a negative w4a16_status_t and launches nothing.
 * M == 0 (or N == 0 for pack) is a valid no-op.  A launch failure returns
 * W4A16_ERR_CUDA.  Faults during execution surface through CUDA as usual.
 * Kernels bound every wait they make; a wait that runs out records
 * W4A16_ERR_TIMEOUT in a device status word read by w4a16_last_device_error.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *w4a16_stream_t;

typedef enum { W4A16_F16 = 0, W4A16_BF16 = 1 } w4a16_dtype_t;

typedef enum {
    W4A16_PATH_AUTO = 0,     /* the dispatcher decides from M and the shape   */
    W4A16_PATH_DECODE = 1,   /* skinny split-K kernel; valid for M <= 8       */
    W4A16_PATH_PREFILL = 2   /* tcgen05 fused-dequant GEMM; any M >= 1        */
} w4a16_path_t;

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_NULL = -1,     /* a required pointer is NULL                    */
    W4A16_ERR_SHAPE = -2,    /* M, N or K out of range / not divisible        */
    W4A16_ERR_GROUP = -3,    /* G not in {32, 64, 128} or K % G != 0          */
    W4A16_ERR_ALIGN = -4,    /* a pointer is not 16-byte aligned              */
    W4A16_ERR_DTYPE = -5,    /* dtype not W4A16_F16 / W4A16_BF16              */
    W4A16_ERR_CUDA = -6,     /* a CUDA runtime call or launch failed          */
    W4A16_ERR_DEVICE = -7,   /* device is not sm_103 / state set-up failed    */
    W4A16_ERR_TIMEOUT = -8,  /* a kernel's bounded wait ran out (device word) */
    W4A16_ERR_ARG = -9       /* other invalid argument (e.g. path enum); in the
                                device status word: an out-of-range expert id */
} w4a16_status_t;

/* Concurrency: the default kernels keep no state between calls, so calls on
 * any streams may overlap.  The balanced decode kernel (an option, see
 * w4a16_debug_set_config which = 4) keeps per-row-block tickets and partial
 * sums in a scratch buffer per stream, made by the first call on that stream
 * with the option on (outside stream capture; during a capture the call
 * falls back to the default decode kernel instead of allocating). */

/* Limits checked by the validation (shapes must also fit in int32 indexing). */
#define W4A16_MAX_DECODE_M 8

/* Pack 4-bit weights.  q: device uint8 [N, K], values 0..15 (higher bits are
 * ignored); qweight: device int32 [N, K/8].  Requires N >= 0, K % 8 == 0.
 * Source: "[ROCm][Kernel] Add HybridW4A16LinearKernel", PR description
 * (weights packed [N, K//8]). */
int w4a16_pack(const uint8_t *q, int N, int K, int32_t *qweight, w4a16_stream_t stream);

/* Pack zero points.  z: device uint8 [N, n_groups], values 0..15;
 * qzeros: device int32 [N/8, n_groups].  Requires N % 8 == 0.
 * Source: "Upstream sync 67/N ... (conflict)", section "Upstream's Python
 * side is kept -- and it does NOT work here" (packed 8 x uint4 along dim 0). */
int w4a16_pack_zeros(const uint8_t *z, int N, int n_groups, int32_t *qzeros,
                     w4a16_stream_t stream);

/* Materialise the dequantised weights: out[n, k] = RN_dtype((q - z) * s),
 * device [N, K] of dtype, k in natural order.  Bit-exact with the definition
 * above.  Runs the register routine of the prefill GEMM kernel (the same
 * code path as w4a16_dequant_debug_ex with W4A16_DQ_PREFILL).  Validation as
 * for w4a16_gemm (G, K % G, N % 8, alignment).
 * Source: "[ROCm][Kernel] Add HybridW4A16LinearKernel", PR description
 * (symmetric bias 8 / per-group zero points; the magic-number dequant). */
int w4a16_dequant_debug(const int32_t *qweight, const void *scales,
                        const int32_t *qzeros_or_null, int G, int N, int K, void *out,
                        w4a16_dtype_t dtype, w4a16_stream_t stream);

/* Which GEMM kernel's dequantisation routine w4a16_dequant_debug_ex runs. */
typedef enum {
    W4A16_DQ_PREFILL = 0,    /* natural (k, k+1) pairs, constants as kernel data       */
    W4A16_DQ_DECODE = 1,     /* (k, k+4) pairs, constants as kernel data (cluster decode) */
    W4A16_DQ_BALANCED = 2    /* (k, k+4) pairs, immediate constants (balanced decode)  */
} w4a16_dq_routine_t;

/* w4a16_dequant_debug with the routine chosen: each GEMM kernel's own
 * dequantisation code, its output put in natural k order, so that a test can
 * hold every routine to the definition bit for bit.  routine outside the enum
 * -> W4A16_ERR_ARG; otherwise as w4a16_dequant_debug.
 * Source: as w4a16_dequant_debug. */
int w4a16_dequant_debug_ex(const int32_t *qweight, const void *scales,
                           const int32_t *qzeros_or_null, int G, int N, int K, void *out,
                           w4a16_dtype_t dtype, w4a16_stream_t stream, int routine);

/* y = x . dequant(W)^T on `stream`.  x, scales and out share `dtype`.
 * Requires M >= 0, N > 0 with N % 8 == 0, K > 0 with K % G == 0,
 * G in {32, 64, 128}, every pointer 16-byte aligned.  Routes M <= threshold
 * to the decode kernel and larger M to the prefill kernel (the threshold is
 * reported by w4a16_select_path).
 * Source: "[ROCm][Kernel] Add HybridW4A16LinearKernel", PR description (M
 * routing between a skinny split-K decode GEMM and a fused-dequant GEMM). */
int w4a16_gemm(const void *x, int M, int K, const int32_t *qweight, const void *scales,
               const int32_t *qzeros_or_null, int G, int N, void *out,
               w4a16_stream_t stream, w4a16_dtype_t dtype);

/* The same call with the dtype fixed by the name. */
int w4a16_gemm_f16(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                   const int32_t *qzeros_or_null, int G, int N, void *out,
                   w4a16_stream_t stream);
int w4a16_gemm_bf16(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                    const int32_t *qzeros_or_null, int G, int N, void *out,
                    w4a16_stream_t stream);

/* w4a16_gemm with the kernel forced: W4A16_PATH_DECODE requires M <= 8
 * (else W4A16_ERR_SHAPE); W4A16_PATH_AUTO is w4a16_gemm. */
int w4a16_gemm_ex(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                  const int32_t *qzeros_or_null, int G, int N, void *out,
                  w4a16_stream_t stream, w4a16_dtype_t dtype, w4a16_path_t path);

/* Epilogues the layer can fuse after its GEMM. */
typedef enum {
    W4A16_EPI_NONE = 0,      /* out [M, N] = y (+ bias)                        */
    W4A16_EPI_SILU_MUL = 1   /* out [M, N/2] = silu(y[:, :N/2]) * y[:, N/2:]   */
} w4a16_epilogue_t;

/* w4a16_gemm_ex with a fused epilogue, in the same launch.
 * Source: "Upstream sync 67/N: merge 382bbd5144 HybridW4A16LinearKernel
 * (conflict)", section "Upstream's Python side is kept -- and it does NOT
 * work here": the skinny GEMM call carries an optional `bias`.  The SiLU-
 * and-multiply epilogue is the step that follows a merged gate/up projection
 * in the models the pages benchmark.
 *  bias_or_null: device [N] in `dtype` (2-byte aligned), added to the fp32
 *    sums before the one rounding, or NULL;
 *  epilogue W4A16_EPI_NONE: out [M, N] = RN(x . dequant(W)^T + bias);
 *  epilogue W4A16_EPI_SILU_MUL: W is a merged gate/up weight, rows 0..N/2-1
 *    the gate and rows N/2..N-1 the up projection; with g, u those halves'
 *    fp32 sums plus bias, out [M, N/2] = RN(silu(g) * u), silu(v) =
 *    v / (1 + exp(-v)).  Runs on the decode kernel only: M must be <=
 *    W4A16_MAX_DECODE_M and path AUTO or DECODE (else W4A16_ERR_SHAPE /
 *    W4A16_ERR_ARG).
 * Other arguments, requirements and errors as w4a16_gemm_ex; an unknown
 * epilogue is W4A16_ERR_ARG. */
int w4a16_gemm_fused(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                     const int32_t *qzeros_or_null, int G, int N, const void *bias_or_null,
                     int epilogue, void *out, w4a16_stream_t stream, w4a16_dtype_t dtype,
                     w4a16_path_t path);

/* MoE grouped skinny GEMM: the decode kernel over routed experts.
 * Source: "Upstream sync 67/N: merge 382bbd5144 HybridW4A16LinearKernel
 * (conflict)", the conflict table's csrc/rocm/ops.h row and the closing
 * section (fused_moe_wvSplitK_int4_gemm: the MoE version of the skinny
 * GEMM).  The pages give only its name; its result here is
 *   out[t, j, :] = x[t, :] . dequant(W_e)^T  (* route_weights[t, j]),
 *   e = expert_ids[t, j], 0 <= t < T, 0 <= j < topk,
 * with each expert's weight as in w4a16_gemm (RN((q - z) s) weights, fp32
 * accumulation, one rounding of the result).
 *  x            device [T, K] activations (`dtype`);
 *  qweight      device [E, N, K/8] int32, the experts' packed weights stacked;
 *  scales       device [E, N, K/G] (`dtype`);
 *  qzeros_or_null  device [E, N/8, K/G] int32, or NULL (symmetric);
 *  expert_ids   device [T, topk] int32 (read by the kernel: it may be the
 *               output of the kernel before it on the stream); an id outside
 *               [0, E) gives a zero output row and W4A16_ERR_ARG in the
 *               device status word (w4a16_last_device_error);
 *  route_weights_or_null  device [T, topk] fp32 factors, or NULL;
 *  out          device [T, topk, N] (`dtype`).
 * Requirements as w4a16_gemm for N, K, G and the 16-byte alignment of x,
 * qweight, scales, qzeros and out (expert_ids and route weights: 4 bytes);
 * T >= 0 (T == 0 is a no-op), topk >= 1, E >= 1; W4A16_ERR_SHAPE beyond
 * int32 index range. */
int w4a16_moe_gemm(const void *x, int T, int K, const int32_t *qweight, const void *scales,
                   const int32_t *qzeros_or_null, int G, int N, int E, const int32_t *expert_ids,
                   int topk, const float *route_weights_or_null, void *out, w4a16_dtype_t dtype,
                   w4a16_stream_t stream);

/* Dequantised prefill cache.  Source: "[ROCm] Converge the two W4A16 linear
 * kernels onto the upstream shell", section "What this does": an optional
 * dequantised copy of the weight that prefill reads with a plain dtype GEMM,
 * while decode keeps reading the int4 weight.
 *
 * w4a16_dequantize: w_out [N, K] (natural order, `dtype`, 16-byte aligned,
 * caller-owned; N * K * 2 bytes) = RN_dtype((q - z) * s) -- the values
 * w4a16_dequant_debug writes, here as the product entry point that builds the
 * cache.  Arguments and errors as w4a16_dequant_debug. */
int w4a16_dequantize(const int32_t *qweight, const void *scales, const int32_t *qzeros_or_null,
                     int G, int N, int K, void *w_out, w4a16_dtype_t dtype, w4a16_stream_t stream);

/* out [M, N] = RN(x . W^T (+ bias)) for a dense weight W [N, K] in `dtype`
 * (e.g. from w4a16_dequantize): the prefill kernel with its weight operand
 * loaded directly into shared memory by TMA (no dequantisation), fp32
 * accumulation in tensor memory.  Requires M >= 0, N > 0 and K > 0 both
 * multiples of 8, x, w, out 16-byte aligned, bias (optional, [N]) 2-byte
 * aligned.  Errors as w4a16_gemm. */
int w4a16_gemm_dense(const void *x, int M, int K, const void *w, int N, const void *bias_or_null,
                     void *out, w4a16_dtype_t dtype, w4a16_stream_t stream);

/* w4a16_gemm with an optional prefill cache: when w_cache_or_null is given
 * and the dispatcher routes M to the prefill path, the call runs
 * w4a16_gemm_dense on the cache; otherwise (decode-sized M, or no cache) it
 * is w4a16_gemm on the int4 weight.  Both give RN((q - z) s)-weight results
 * within the same tolerance (the cache holds exactly those weights). */
int w4a16_gemm_cached(const void *x, int M, int K, const int32_t *qweight, const void *scales,
                      const int32_t *qzeros_or_null, int G, int N, const void *w_cache_or_null,
                      void *out, w4a16_stream_t stream, w4a16_dtype_t dtype);

/* One layer of a chain (w4a16_gemm_chain): its weights, optional bias,
 * epilogue and output buffer.  N, K and G as in w4a16_gemm. */
typedef struct {
    const int32_t *qweight;
    const void *scales;
    const int32_t *qzeros_or_null;
    const void *bias_or_null;
    int G, N, K;
    int epilogue;            /* w4a16_epilogue_t */
    void *out;               /* [M, N] or, with W4A16_EPI_SILU_MUL, [M, N/2] */
} w4a16_layer_t;

/* A stream of linear layers in which layer i's output is layer i+1's input:
 * layer 0 reads x [M, layers[0].K]; layer i > 0 reads layers[i-1].out, so
 * layers[i].K must equal layer i-1's output width (W4A16_ERR_SHAPE
 * otherwise).  Each layer runs as w4a16_gemm_fused with path AUTO, enqueued
 * back to back on `stream` with programmatic dependent launch: a layer's
 * kernel may start while the previous one drains, streaming its own weights,
 * and reads its input only after the previous kernel has completed.  No
 * weight, scale, zero-point or bias buffer of the chain may be an output of
 * it.  Safe to capture in a CUDA graph.  Source: "[ROCm][Kernel] Add
 * HybridW4A16LinearKernel: Triton prefill + HIP skinny decode", benchmark
 * tables (per-token decode latency over a model's layer stream).  All
 * arguments are checked before the first launch; an error then returns
 * without enqueuing anything. */
int w4a16_gemm_chain(const void *x, int M, const w4a16_layer_t *layers, int n_layers,
                     w4a16_dtype_t dtype, w4a16_stream_t stream);

/* End-to-end form: x_host and out_host are HOST buffers (pinned for full
 * speed); x_dev [M, K] and out_dev [M, N] are caller-owned device staging
 * buffers.  Copies x to the device, runs w4a16_gemm, copies y back and
 * synchronises `stream` before returning. */
int w4a16_gemm_host(const void *x_host, int M, int K, const int32_t *qweight,
                    const void *scales, const int32_t *qzeros_or_null, int G, int N,
                    void *out_host, w4a16_dtype_t dtype, void *x_dev, void *out_dev,
                    w4a16_stream_t stream);

/* w4a16_gemm_host without the synchronisation: the copy in, the GEMM and
 * the copy out are enqueued on `stream` and the call returns; out_host holds
 * y once the stream has reached that point (the caller synchronises, e.g.
 * once after a whole step of layers).  x_host and out_host must stay valid
 * and unchanged until then; pinned host memory makes the copies
 * asynchronous. */
int w4a16_gemm_host_async(const void *x_host, int M, int K, const int32_t *qweight,
                          const void *scales, const int32_t *qzeros_or_null, int G, int N,
                          void *out_host, w4a16_dtype_t dtype, void *x_dev, void *out_dev,
                          w4a16_stream_t stream);

/* Host-only: which kernel w4a16_gemm would run (W4A16_PATH_DECODE or
 * W4A16_PATH_PREFILL), or a negative status for invalid arguments.  sym != 0
 * means qzeros_or_null == NULL. */
int w4a16_select_path(int M, int N, int K, int G, int sym, int dtype);

/* Test hook: the prefill launch plan the dispatcher would pick for an
 * M x N x K problem (dense != 0: the dense form) on a device with sm_count
 * SMs whose prefill kernel keeps clusters[k - 1] clusters of k CTAs resident
 * at once (k = 1..8, as the occupancy query reports).  Host arithmetic only:
 * no device is touched.  out (13 ints, caller-owned) receives n_split (N
 * when the plan is one launch), then for the first and the second launch
 * {BN, x-ring stages, dequantised-weight stages, packed-weight stages, KS,
 * swapped operands (0/1)}.  Returns W4A16_OK, or W4A16_ERR_ARG for a
 * non-positive or misaligned shape, sm_count <= 0, a negative cluster count
 * or a NULL pointer. */
int w4a16_debug_prefill_plan(int M, int N, int K, int dense, int sm_count, const int *clusters, int *out);

/* Profiling hook: a per-CTA timeline of the decode kernel.  trace_buf
 * (device memory, 8-byte aligned, caller-owned, 4 x 512 x 8 uint64 =
 * 131072 bytes, zeroed by the caller) receives, for every CTA c < 512 of a
 * decode launch whose (N, K) is pair i of nk (8 ints: up to four (N, K)
 * pairs; unused pairs 0), at [i][c][e] the %globaltimer value in ns of event
 * e: 0 entry, 1 grid-dependency wait returned, 2 x staged, 3 first weight
 * stage ready, 4 loop end, 5 cluster partials gathered (cluster rank 0
 * only), 6 exit; [i][c][7] is the CTA's cluster rank.  The buffer travels
 * in the launch parameters, so the setting applies to launches made (and
 * CUDA graphs captured) after this call; a graph captured before it keeps
 * the setting it was captured with.  Each launch of a traced layer
 * overwrites its entries (the last one wins); MoE launches are not traced.
 * trace_buf = NULL turns the trace off (the default).  The buffer must
 * outlive every launch and graph that writes it.  Host state, not
 * thread-safe against concurrent launches.  The stamps exist only in the
 * trace build of the library (compiled with W4A16_DECODE_TRACE defined,
 * libw4a16_trace.so); the default build's decode kernel has none, and there
 * any non-NULL trace_buf returns W4A16_ERR_ARG.  Returns W4A16_OK,
 * W4A16_ERR_ARG (nk NULL, a misaligned buffer, or a buffer given to the
 * default build) or W4A16_ERR_DEVICE. */
int w4a16_debug_decode_trace(unsigned long long *trace_buf_or_null, const int *nk);

/* The decode GEMM (M <= 8) without any device allocation, ever.  The pages
 * have no counterpart of this entry point: it is a library addition for
 * callers that must not allocate device memory after start-up (an engine
 * that reserves its whole device arena up front, or code where a cudaMalloc
 * would synchronise the device or is not allowed).  Arguments, layouts and
 * host-side validation are those of w4a16_gemm; the result is that of the
 * balanced decode kernel (debug configuration which = 4).  The kernel's
 * scratch is static device memory of fixed size, so: M must be 0..8 and N at
 * most 131072, and the staged x (M x K values) plus the kernel's partial
 * slots must fit in its 220 KB of shared memory (for example M = 8 with
 * K = 14336 does not) -- W4A16_ERR_SHAPE otherwise; the device may have at
 * most 256 SMs (W4A16_ERR_DEVICE).  The first call on a device, with that
 * device current, sets the scratch up (looks up its address and clears it);
 * make that first call before any stream capture: made during a capture it
 * returns W4A16_ERR_DEVICE and touches nothing, and the next call outside a
 * capture sets up as usual (a failed set-up is retried).  Programmatic
 * dependent launch follows the same switch as w4a16_gemm.  All calls on a
 * device share the scratch: calls whose kernels overlap on the GPU race on
 * it; calls in order on one stream are safe. */
int w4a16_gemm_decode_noalloc(const void *x, int M, int K, const int32_t *qweight,
                              const void *scales, const int32_t *qzeros_or_null, int G, int N,
                              void *out, w4a16_stream_t stream, w4a16_dtype_t dtype);

/* Device status word of the current device: W4A16_OK, or W4A16_ERR_TIMEOUT
 * if a kernel gave up a bounded wait since the last clear.  Synchronises the
 * device to read it. */
int w4a16_last_device_error(void);
int w4a16_clear_device_error(void);

/* ABI version (major * 100 + minor). */
int w4a16_version(void);

/* Tuning hook (process-wide, for benchmarks and sweeps).  which = 1: decode
 * configuration vals = {R, NW, NB, NS, S} (16-row blocks per warp, warps per
 * CTA, 128-wide TMA boxes per ring stage, ring stages, cluster CTAs along
 * K), n = 5;
 * which = 2: prefill configuration vals = {BN, x-ring stages, dequantised-
 * weight stages, packed-weight stages[, KS]}, n = 4 or 5 (BN a multiple of
 * 16 in [16, 256]; the rings must fit in shared memory, for the fused
 * kernel or for the dense form, which has no packed-weight ring and ignores
 * that entry; KS = CTAs of a cluster splitting K, 0 or absent = chosen per
 * call, else 1..8, lowered to the number of 256-k weight tiles; KS > 1
 * needs the fp32 partial tile, BN KB, to fit over the rings).  While set,
 * every prefill call runs as one launch with it, and a call whose kernel
 * it does not fit returns W4A16_ERR_ARG;
 * which = 3: programmatic dependent launch on/off, vals = {flag}, n = 1;
 * which = 4: balanced decode kernel vals = {on (1) / off (0), load ring
 * depth in units (2, 4 or 6)}, n = 2;
 * which = 8: test of the prefill row split, vals = {n_split}, n = 1 (a
 * positive multiple of 256): every prefill call (fused or dense form) with
 * N > n_split runs as two launches, weight rows [0, n_split) and
 * [n_split, N), each with the configuration the dispatcher picks for it
 * (unless which = 2 is set); n = 0 turns it off;
 * which = 7: test of the timeout path, vals = {on (1) / off (0)}, n = 1:
 * while on, the decode kernel issues no weight copies, so every CTA's bounded
 * wait for them runs out (about 2 s), the kernel leaves without touching
 * memory beyond its own output and records W4A16_ERR_TIMEOUT in the status
 * word (its output is then meaningless); n = 0 turns it off;
 * n = 0 restores the built-in choice for which = 1, 2, 4 or 8.  An invalid
 * configuration is rejected here or, for the decode shape limits, by the
 * next w4a16_gemm call with W4A16_ERR_ARG. */
int w4a16_debug_set_config(int which, const int *vals, int n);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
