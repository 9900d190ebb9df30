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
    return os.path.join(_HERE, _LIBNAME)


def load_library():
    """Load libw4a16.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with w4a16_group_quantised_gb300.build.build()")
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
            "w4a16_gemm_host": [P, I, I, P, P, P, I, I, P, I, P, P, P],
            "w4a16_gemm_decode_noalloc": [P, I, I, P, P, P, I, I, P, P, I],
            "w4a16_select_path": [I, I, I, I, I, I],
            "w4a16_last_device_error": [],
            "w4a16_clear_device_error": [],
            "w4a16_version": [],
            "w4a16_debug_set_config": [I, P, I],
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
    _require_int32("qweight", qweight)
    _require_int32("qzeros", qzeros)
    M, K = x.shape
    N = qweight.shape[0]
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


def w4a16_gemm_decode_noalloc(x, qweight, scales, qzeros, G: int, out=None, stream=None):
    """y = x . dequant(W)^T for M <= 8 through the allocation-free entry point
    (static device scratch; see include/w4a16.h).  `out` must be given by a
    caller that must not allocate; if it is None a tensor is created here."""
    import torch
    lib = load_library()
    _require_int32("qzeros", qzeros)
    _require_int32("qweight", qweight)
    M, K = x.shape
    N = qweight.shape[0]
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
    kernel {on, ring depth}.  vals=None restores the built-in choice."""
    lib = load_library()
    if vals is None:
        rc = lib.w4a16_debug_set_config(which, None, 0)
    else:
        arr = (ctypes.c_int * len(vals))(*[int(v) for v in vals])
        rc = lib.w4a16_debug_set_config(which, arr, len(vals))
    _check("w4a16_debug_set_config", rc)


def w4a16_last_device_error() -> int:
    """Status word written by kernels whose bounded waits ran out (0 = none)."""
    return load_library().w4a16_last_device_error()
