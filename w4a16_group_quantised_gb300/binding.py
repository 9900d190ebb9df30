"""Thin ctypes binding of libw4a16.so (argument marshalling only).

Every function has the name of the C entry point it calls.  Tensors are torch
CUDA tensors; their data pointers and the current CUDA stream are handed to
the library unchanged.  No arithmetic of the layer happens here, and there is
no fallback: if the library cannot be loaded every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBNAME = "libw4a16.so"
_lock = threading.Lock()
_lib = None

W4A16_F16, W4A16_BF16 = 0, 1
PATH_AUTO, PATH_DECODE, PATH_PREFILL = 0, 1, 2
EPI_NONE, EPI_SILU_MUL = 0, 1

_STATUS = {
    0: "W4A16_OK", -1: "W4A16_ERR_NULL", -2: "W4A16_ERR_SHAPE", -3: "W4A16_ERR_GROUP",
    -4: "W4A16_ERR_ALIGN", -5: "W4A16_ERR_DTYPE", -6: "W4A16_ERR_CUDA",
    -7: "W4A16_ERR_DEVICE", -8: "W4A16_ERR_TIMEOUT", -9: "W4A16_ERR_ARG",
}


class W4A16Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({_STATUS.get(code, 'unknown')})")
        self.code = code


def library_path() -> str:
    """libw4a16.so, or with W4A16_LIBRARY=trace the profiling build
    libw4a16_trace.so (the decode kernel's timeline stamps compiled in)."""
    v = os.environ.get("W4A16_LIBRARY", "")
    if v not in ("", "trace"):
        raise ValueError(f"W4A16_LIBRARY={v!r}: expected unset or 'trace'")
    return os.path.join(_HERE, "libw4a16_trace.so" if v == "trace" else _LIBNAME)


def load_library():
    """Load the library (library_path()); raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with w4a16_group_quantised_gb300.build.build()"
                + (" (variant='trace')" if path.endswith("_trace.so") else ""))
        lib = ctypes.CDLL(path)
        P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        sig = {
            "w4a16_pack": [P, I, I, P, P],
            "w4a16_pack_zeros": [P, I, I, P, P],
            "w4a16_dequant_debug": [P, P, P, I, I, I, P, I, P],
            "w4a16_dequant_debug_ex": [P, P, P, I, I, I, P, I, P, I],
            "w4a16_gemm": [P, I, I, P, P, P, I, I, P, P, I],
            "w4a16_gemm_f16": [P, I, I, P, P, P, I, I, P, P],
            "w4a16_gemm_bf16": [P, I, I, P, P, P, I, I, P, P],
            "w4a16_gemm_ex": [P, I, I, P, P, P, I, I, P, P, I, I],
            "w4a16_gemm_fused": [P, I, I, P, P, P, I, I, P, I, P, P, I, I],
            "w4a16_gemm_chain": [P, I, P, I, I, P],
            "w4a16_dequantize": [P, P, P, I, I, I, P, I, P],
            "w4a16_moe_gemm": [P, I, I, P, P, P, I, I, I, P, I, P, P, I, P],
            "w4a16_gemm_dense": [P, I, I, P, I, P, P, I, P],
            "w4a16_gemm_cached": [P, I, I, P, P, P, I, I, P, P, P, I],
            "w4a16_gemm_host": [P, I, I, P, P, P, I, I, P, I, P, P, P],
            "w4a16_gemm_host_async": [P, I, I, P, P, P, I, I, P, I, P, P, P],
            "w4a16_gemm_decode_noalloc": [P, I, I, P, P, P, I, I, P, P, I],
            "w4a16_select_path": [I, I, I, I, I, I],
            "w4a16_last_device_error": [],
            "w4a16_clear_device_error": [],
            "w4a16_version": [],
            "w4a16_debug_set_config": [I, P, I],
            "w4a16_debug_prefill_plan": [I, I, I, I, I, P, P],
            "w4a16_debug_decode_trace": [P, P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I
        _lib = lib
        return lib


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise W4A16Error(fn, code)


def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return W4A16_F16
    if t.dtype == torch.bfloat16:
        return W4A16_BF16
    raise TypeError(f"activation dtype must be float16 or bfloat16, got {t.dtype}")


def _require_int32(name, t):
    import torch
    if t is not None and t.dtype not in (torch.int32,):
        # The packed zero-point contract: int32, 8 x uint4 along dim 0.
        raise TypeError(f"{name} must be int32 (packed 8 x uint4), got {t.dtype}")


def _check_gemm_operands(x, qweight, scales, qzeros, G, out, out_cols=None, bias=None,
                         require_cuda=True):
    """Host-side checks of the operands' types, dtypes, shapes, layout and
    device before the C call (which checks again what it can see: sizes,
    alignment, G).  TypeError for a wrong type or dtype, ValueError for a
    wrong shape, layout or device."""
    import torch
    named = [("x", x), ("qweight", qweight), ("scales", scales), ("qzeros", qzeros), ("out", out),
             ("bias", bias)]
    for name, t in named:
        if t is None and name in ("qzeros", "out", "bias"):
            continue
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
        if require_cuda and t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor, got device {t.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    devs = {t.device for _, t in named if t is not None}
    if len(devs) > 1:
        raise ValueError(f"operands are on different devices: {sorted(map(str, devs))}")
    if not isinstance(G, int) or isinstance(G, bool):
        raise TypeError(f"G must be an int, got {type(G).__name__}")
    _dtype_code(x)
    _require_int32("qweight", qweight)
    _require_int32("qzeros", qzeros)
    if x.dim() != 2 or qweight.dim() != 2 or scales.dim() != 2:
        raise ValueError("x, qweight and scales must be 2-D")
    M, K = x.shape
    N = qweight.shape[0]
    if qweight.shape[1] * 8 != K:
        raise ValueError(f"qweight must be [N, K/8] = [{N}, {K // 8}], got {list(qweight.shape)}")
    if scales.dtype != x.dtype:
        raise TypeError(f"scales dtype {scales.dtype} differs from x dtype {x.dtype}")
    if G > 0 and K % G == 0 and list(scales.shape) != [N, K // G]:
        raise ValueError(f"scales must be [N, K/G] = [{N}, {K // G}], got {list(scales.shape)}")
    if qzeros is not None and G > 0 and K % G == 0 and list(qzeros.shape) != [N // 8, K // G]:
        raise ValueError(f"qzeros must be [N/8, K/G] = [{N // 8}, {K // G}], got {list(qzeros.shape)}")
    if bias is not None:
        if bias.dtype != x.dtype:
            raise TypeError(f"bias dtype {bias.dtype} differs from x dtype {x.dtype}")
        if bias.dim() != 1 or bias.shape[0] != N:
            raise ValueError(f"bias must be [N] = [{N}], got {list(bias.shape)}")
    if out is not None:
        cols = N if out_cols is None else out_cols
        if out.dtype != x.dtype:
            raise TypeError(f"out dtype {out.dtype} differs from x dtype {x.dtype}")
        if list(out.shape) != [M, cols]:
            raise ValueError(f"out must be [{M}, {cols}], got {list(out.shape)}")
    return M, K, N


def w4a16_pack(q, qweight=None, stream=None):
    """q uint8 [N, K] (values 0..15) -> qweight int32 [N, K/8]."""
    import torch
    N, K = q.shape
    if qweight is None:
        qweight = torch.empty((N, K // 8), dtype=torch.int32, device=q.device)
    lib = load_library()
    _check("w4a16_pack", lib.w4a16_pack(_p(q), N, K, _p(qweight), _stream_ptr(stream)))
    return qweight


def w4a16_pack_zeros(z, qzeros=None, stream=None):
    """z uint8 [N, n_groups] (values 0..15) -> qzeros int32 [N/8, n_groups]."""
    import torch
    N, ng = z.shape
    if qzeros is None:
        qzeros = torch.empty((N // 8, ng), dtype=torch.int32, device=z.device)
    lib = load_library()
    _check("w4a16_pack_zeros", lib.w4a16_pack_zeros(_p(z), N, ng, _p(qzeros), _stream_ptr(stream)))
    return qzeros


DQ_PREFILL, DQ_DECODE, DQ_BALANCED = 0, 1, 2


def w4a16_dequant_debug(qweight, scales, qzeros, G: int, out=None, stream=None, routine=None):
    """Materialise RN_dtype((q - z) * s) as a [N, K] tensor of the scales' dtype
    (routine: None = w4a16_dequant_debug, else the w4a16_dequant_debug_ex routine)."""
    import torch
    _require_int32("qweight", qweight)
    _require_int32("qzeros", qzeros)
    N, K8 = qweight.shape
    K = K8 * 8
    dt = _dtype_code(scales)
    if out is None:
        out = torch.empty((N, K), dtype=scales.dtype, device=qweight.device)
    lib = load_library()
    if routine is None:
        rc = lib.w4a16_dequant_debug(_p(qweight), _p(scales), _p(qzeros), G, N, K, _p(out), dt,
                                     _stream_ptr(stream))
    else:
        rc = lib.w4a16_dequant_debug_ex(_p(qweight), _p(scales), _p(qzeros), G, N, K, _p(out), dt,
                                        _stream_ptr(stream), routine)
    _check("w4a16_dequant_debug", rc)
    return out


def w4a16_gemm(x, qweight, scales, qzeros, G: int, out=None, stream=None, path: int = PATH_AUTO):
    """y[M, N] = x[M, K] . dequant(W)^T in the dtype of x."""
    import torch
    M, K, N = _check_gemm_operands(x, qweight, scales, qzeros, G, out)
    dt = _dtype_code(x)
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    lib = load_library()
    if path == PATH_AUTO:
        rc = lib.w4a16_gemm(_p(x), M, K, _p(qweight), _p(scales), _p(qzeros), G, N, _p(out),
                            _stream_ptr(stream), dt)
    else:
        rc = lib.w4a16_gemm_ex(_p(x), M, K, _p(qweight), _p(scales), _p(qzeros), G, N, _p(out),
                               _stream_ptr(stream), dt, path)
    _check("w4a16_gemm", rc)
    return out


def w4a16_gemm_fused(x, qweight, scales, qzeros, G: int, bias=None, epilogue: int = EPI_NONE,
                     out=None, stream=None, path: int = PATH_AUTO):
    """x . dequant(W)^T + bias with the epilogue fused: EPI_NONE gives [M, N];
    EPI_SILU_MUL (W = [gate; up], N = 2 I) gives silu(gate) * up, [M, I]."""
    import torch
    if epilogue not in (EPI_NONE, EPI_SILU_MUL):
        raise ValueError(f"unknown epilogue {epilogue}")
    N0 = qweight.shape[0] if isinstance(qweight, torch.Tensor) else 0
    cols = N0 // 2 if epilogue == EPI_SILU_MUL else N0
    M, K, N = _check_gemm_operands(x, qweight, scales, qzeros, G, out, out_cols=cols, bias=bias)
    if epilogue == EPI_SILU_MUL and N % 2:
        raise ValueError("SiLU-and-multiply needs an even number of weight rows")
    dt = _dtype_code(x)
    if out is None:
        out = torch.empty((M, cols), dtype=x.dtype, device=x.device)
    lib = load_library()
    rc = lib.w4a16_gemm_fused(_p(x), M, K, _p(qweight), _p(scales), _p(qzeros), G, N, _p(bias), epilogue,
                              _p(out), _stream_ptr(stream), dt, path)
    _check("w4a16_gemm_fused", rc)
    return out


def w4a16_moe_gemm(x, qweight, scales, qzeros, G: int, expert_ids, route_weights=None, out=None, stream=None):
    """MoE grouped skinny GEMM: out [T, topk, N] with out[t, j] = x[t] .
    dequant(W_{expert_ids[t, j]})^T (* route_weights[t, j]); qweight
    [E, N, K/8], scales [E, N, K/G], qzeros [E, N/8, K/G] or None."""
    import torch
    for name, t in (("x", x), ("qweight", qweight), ("scales", scales), ("qzeros", qzeros),
                    ("expert_ids", expert_ids), ("route_weights", route_weights), ("out", out)):
        if t is not None and (not isinstance(t, torch.Tensor) or t.device.type != "cuda" or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    _require_int32("qweight", qweight)
    _require_int32("qzeros", qzeros)
    dt = _dtype_code(x)
    if scales.dtype != x.dtype:
        raise TypeError("scales must have the dtype of x")
    if expert_ids.dtype != torch.int32 or expert_ids.dim() != 2:
        raise TypeError("expert_ids must be int32 [T, topk]")
    if route_weights is not None and (route_weights.dtype != torch.float32
                                      or route_weights.shape != expert_ids.shape):
        raise TypeError("route_weights must be float32 [T, topk]")
    T, K = x.shape
    E, N, K8 = qweight.shape
    topk = expert_ids.shape[1]
    if K8 * 8 != K or expert_ids.shape[0] != T:
        raise ValueError("qweight must be [E, N, K/8] and expert_ids [T, topk]")
    if G > 0 and K % G == 0 and list(scales.shape) != [E, N, K // G]:
        raise ValueError(f"scales must be [E, N, K/G] = [{E}, {N}, {K // G}]")
    if qzeros is not None and G > 0 and K % G == 0 and list(qzeros.shape) != [E, N // 8, K // G]:
        raise ValueError(f"qzeros must be [E, N/8, K/G] = [{E}, {N // 8}, {K // G}]")
    if out is None:
        out = torch.empty((T, topk, N), dtype=x.dtype, device=x.device)
    elif list(out.shape) != [T, topk, N] or out.dtype != x.dtype:
        raise ValueError(f"out must be [{T}, {topk}, {N}] of x's dtype")
    rc = load_library().w4a16_moe_gemm(_p(x), T, K, _p(qweight), _p(scales), _p(qzeros), G, N, E, _p(expert_ids),
                                       topk, _p(route_weights), _p(out), dt, _stream_ptr(stream))
    _check("w4a16_moe_gemm", rc)
    return out


def w4a16_dequantize(qweight, scales, qzeros, G: int, out=None, stream=None):
    """The dequantised prefill cache: W [N, K] = RN_dtype((q - z) * s) in the
    scales' dtype (natural order)."""
    import torch
    _require_int32("qweight", qweight)
    _require_int32("qzeros", qzeros)
    N, K8 = qweight.shape
    K = K8 * 8
    if out is None:
        out = torch.empty((N, K), dtype=scales.dtype, device=qweight.device)
    rc = load_library().w4a16_dequantize(_p(qweight), _p(scales), _p(qzeros), G, N, K, _p(out),
                                         _dtype_code(scales), _stream_ptr(stream))
    _check("w4a16_dequantize", rc)
    return out


def w4a16_gemm_dense(x, w, bias=None, out=None, stream=None):
    """out [M, N] = x . W^T (+ bias) for a dense weight W [N, K] of x's dtype."""
    import torch
    for name, t in (("x", x), ("w", w), ("bias", bias), ("out", out)):
        if t is not None and (not isinstance(t, torch.Tensor) or t.device.type != "cuda" or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    dt = _dtype_code(x)
    if w.dtype != x.dtype or (bias is not None and bias.dtype != x.dtype):
        raise TypeError("w and bias must have the dtype of x")
    M, K = x.shape
    N = w.shape[0]
    if w.dim() != 2 or w.shape[1] != K:
        raise ValueError(f"w must be [N, {K}], got {list(w.shape)}")
    if bias is not None and list(bias.shape) != [N]:
        raise ValueError(f"bias must be [{N}]")
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    elif list(out.shape) != [M, N] or out.dtype != x.dtype:
        raise ValueError(f"out must be [{M}, {N}] of x's dtype")
    rc = load_library().w4a16_gemm_dense(_p(x), M, K, _p(w), N, _p(bias), _p(out), dt, _stream_ptr(stream))
    _check("w4a16_gemm_dense", rc)
    return out


def w4a16_gemm_cached(x, qweight, scales, qzeros, G: int, w_cache=None, out=None, stream=None):
    """w4a16_gemm, except that prefill-sized M reads the dequantised cache
    w_cache [N, K] (if given) through w4a16_gemm_dense."""
    import torch
    M, K, N = _check_gemm_operands(x, qweight, scales, qzeros, G, out)
    if w_cache is not None and (w_cache.dtype != x.dtype or list(w_cache.shape) != [N, K]
                                or not w_cache.is_contiguous() or w_cache.device != x.device):
        raise ValueError(f"w_cache must be a contiguous [{N}, {K}] tensor of x's dtype on x's device")
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    rc = load_library().w4a16_gemm_cached(_p(x), M, K, _p(qweight), _p(scales), _p(qzeros), G, N, _p(w_cache),
                                          _p(out), _stream_ptr(stream), _dtype_code(x))
    _check("w4a16_gemm_cached", rc)
    return out


class w4a16_layer_t(ctypes.Structure):
    """Mirror of the C struct w4a16_layer_t (include/w4a16.h)."""
    _fields_ = [("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("qzeros_or_null", ctypes.c_void_p), ("bias_or_null", ctypes.c_void_p),
                ("G", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("epilogue", ctypes.c_int), ("out", ctypes.c_void_p)]


def w4a16_gemm_chain(x, layers, stream=None):
    """Run layers back to back, layer i's output feeding layer i+1.  `layers`
    is a sequence of dicts with qweight, scales, qzeros, G and optionally bias,
    epilogue and out (created when missing).  Returns the list of outputs."""
    import torch
    M = x.shape[0]
    outs, structs, inp = [], [], x
    for i, L in enumerate(layers):
        epi = L.get("epilogue", EPI_NONE)
        N = L["qweight"].shape[0]
        cols = N // 2 if epi == EPI_SILU_MUL else N
        out = L.get("out")
        if out is None:
            out = torch.empty((M, cols), dtype=x.dtype, device=x.device)
        _check_gemm_operands(inp, L["qweight"], L["scales"], L.get("qzeros"), L["G"], out, out_cols=cols,
                             bias=L.get("bias"))
        structs.append(w4a16_layer_t(_p(L["qweight"]), _p(L["scales"]), _p(L.get("qzeros")), _p(L.get("bias")),
                                     L["G"], N, inp.shape[1], epi, _p(out)))
        outs.append(out)
        inp = out
    arr = (w4a16_layer_t * max(1, len(structs)))(*structs)
    lib = load_library()
    rc = lib.w4a16_gemm_chain(_p(x), M, ctypes.cast(arr, ctypes.c_void_p), len(structs), _dtype_code(x),
                              _stream_ptr(stream))
    _check("w4a16_gemm_chain", rc)
    return outs


def w4a16_gemm_host(x_host, qweight, scales, qzeros, G: int, out_host, dev_x, dev_out,
                    stream=None):
    """End-to-end call: x from pinned host memory, y back to host memory.

    x_host / out_host are pinned CPU tensors; dev_x / dev_out are device
    staging buffers of the same shapes (the caller owns all four)."""
    M, K = x_host.shape
    N = qweight.shape[0]
    dt = _dtype_code(x_host)
    lib = load_library()
    rc = lib.w4a16_gemm_host(_p(x_host), M, K, _p(qweight), _p(scales), _p(qzeros), G, N,
                             _p(out_host), dt, _p(dev_x), _p(dev_out), _stream_ptr(stream))
    _check("w4a16_gemm_host", rc)
    return out_host


def w4a16_gemm_host_async(x_host, qweight, scales, qzeros, G: int, out_host, dev_x, dev_out, stream=None):
    """w4a16_gemm_host without the synchronisation: copies and GEMM are
    enqueued on the stream; out_host is valid once the stream is synchronised."""
    M, K = x_host.shape
    N = qweight.shape[0]
    dt = _dtype_code(x_host)
    rc = load_library().w4a16_gemm_host_async(_p(x_host), M, K, _p(qweight), _p(scales), _p(qzeros), G, N,
                                              _p(out_host), dt, _p(dev_x), _p(dev_out), _stream_ptr(stream))
    _check("w4a16_gemm_host_async", rc)
    return out_host


def w4a16_gemm_decode_noalloc(x, qweight, scales, qzeros, G: int, out=None, stream=None):
    """y = x . dequant(W)^T for M <= 8 through the allocation-free entry point
    (static device scratch; see include/w4a16.h).  `out` must be given by a
    caller that must not allocate; if it is None a tensor is created here."""
    import torch
    lib = load_library()
    M, K, N = _check_gemm_operands(x, qweight, scales, qzeros, G, out)
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    rc = lib.w4a16_gemm_decode_noalloc(_p(x), M, K, _p(qweight), _p(scales),
                                       _p(qzeros) if qzeros is not None else None, G, N, _p(out),
                                       _stream_ptr(stream), _dtype_code(x))
    _check("w4a16_gemm_decode_noalloc", rc)
    return out


def w4a16_select_path(M: int, N: int, K: int, G: int, sym: bool, dtype: int) -> int:
    """Which kernel the dispatcher picks: 1 = decode, 2 = prefill (host logic only)."""
    return load_library().w4a16_select_path(M, N, K, G, 1 if sym else 0, dtype)


def w4a16_debug_set_config(which: int, vals=None) -> None:
    """Tuning hook (see include/w4a16.h): which=1 cluster decode kernel
    {R, NW, NB, NS, S}; which=2 prefill {BN, x stages, A stages, W stages[, KS]};
    which=3 programmatic dependent launch {flag}; which=4 balanced decode
    kernel {on, ring depth}; which=7 timeout-path test {on} (decode kernels
    issue no weight copies, so their bounded waits run out); which=8 prefill
    row split (fused and dense forms) at {n_split} (a multiple of 256).  vals=None
    restores the built-in choice."""
    lib = load_library()
    if vals is None:
        rc = lib.w4a16_debug_set_config(which, None, 0)
    else:
        arr = (ctypes.c_int * len(vals))(*[int(v) for v in vals])
        rc = lib.w4a16_debug_set_config(which, arr, len(vals))
    _check("w4a16_debug_set_config", rc)


TRACE_LAYERS, TRACE_CTAS, TRACE_EVENTS = 4, 512, 8


def w4a16_debug_decode_trace(shapes=None):
    """Profiling hook (see include/w4a16.h), in the trace build of the
    library only (W4A16_LIBRARY=trace): with shapes = up to four (N, K)
    pairs, every later decode launch of such a layer writes its per-CTA
    timeline into a device buffer, which is returned ([4, 512, 8] int64:
    %globaltimer ns of entry, release, x staged, first stage, loop end,
    gather, exit, then the cluster rank; zero where no CTA wrote).
    shapes=None turns the trace off and returns None.  The default library
    raises W4A16Error (W4A16_ERR_ARG) for a non-None shapes."""
    import torch
    lib = load_library()
    if shapes is None:
        _check("w4a16_debug_decode_trace", lib.w4a16_debug_decode_trace(None, None))
        return None
    if not 1 <= len(shapes) <= TRACE_LAYERS:
        raise ValueError("w4a16_debug_decode_trace: one to four (N, K) pairs")
    nk = [0] * (2 * TRACE_LAYERS)
    for i, (n, k) in enumerate(shapes):
        nk[2 * i], nk[2 * i + 1] = int(n), int(k)
    buf = torch.zeros((TRACE_LAYERS, TRACE_CTAS, TRACE_EVENTS), dtype=torch.int64, device="cuda")
    arr = (ctypes.c_int * len(nk))(*nk)
    _check("w4a16_debug_decode_trace", lib.w4a16_debug_decode_trace(ctypes.c_void_p(buf.data_ptr()), arr))
    return buf


def w4a16_last_device_error() -> int:
    """Status word written by kernels whose bounded waits ran out (0 = none)."""
    return load_library().w4a16_last_device_error()


def w4a16_clear_device_error() -> None:
    """Synchronise the device and reset the status word (and the balanced
    decode kernel's tickets) after a timeout."""
    _check("w4a16_clear_device_error", load_library().w4a16_clear_device_error())
