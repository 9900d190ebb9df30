"""CPU oracle for the W4A16 group-quantised linear layer (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library.  The arithmetic
lives in ``oracle.c`` (plain C, binary64); this module builds it with gcc and
wraps it with ctypes, plus one independent numpy restatement used to
cross-check the C code on small inputs (``np_*`` functions).

Sources the oracle follows (page titles, not files):
  * "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP skinny
    decode", PR description: packed [N, K/8] weights, uint4b8 symmetric
    (bias 8) or per-group zero points, G in {32, 64, 128}.
  * "Upstream sync 67/N: merge 382bbd5144 HybridW4A16LinearKernel (conflict)",
    section "Upstream's Python side is kept -- and it does NOT work here":
    zero points packed int32 [N/8, groups], 8 x uint4 along dim 0.

Parity pins: see tests/test_oracle_pins.py.  Every public function here is
pinned there; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (OpenMP over output columns)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16, I]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_double_to_half.argtypes = [ctypes.c_double, I]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_pack.argtypes = [P, I, I, P]
            lib.oracle_unpack.argtypes = [P, I, I, P]
            lib.oracle_pack_zeros.argtypes = [P, I, I, P]
            lib.oracle_unpack_zeros.argtypes = [P, I, I, P]
            lib.oracle_dequant.argtypes = [P, P, P, I, I, I, I, P]
            lib.oracle_round_products.argtypes = [P, I, I, P]
            lib.oracle_gemm_rows.argtypes = [P, I, I, P, P, P, I, I, I, P, I, I, P]
            lib.oracle_round_array.argtypes = [P, ctypes.c_longlong, I, P]
            lib.oracle_half_array_to_double.argtypes = [P, ctypes.c_longlong, I, P]
            lib.oracle_num_threads.restype = I
            lib.oracle_epilogue.argtypes = [P, I, I, P, I, I, P]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars
def half_to_double(bits: int, dtype: int) -> float:
    return _load().oracle_half_to_double(int(bits), dtype)


def double_to_half(v: float, dtype: int) -> int:
    return _load().oracle_double_to_half(float(v), dtype)


def bits_to_float64(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact values of an array of 16-bit patterns (via the C decoder)."""
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_half_array_to_double(_ptr(b), b.size, dtype, _ptr(out))
    return out


def round_array(v: np.ndarray, dtype: int) -> np.ndarray:
    """RN-even rounding of float64 values to the 16-bit format (bit patterns)."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_array(_ptr(v), v.size, dtype, _ptr(out))
    return out


# ---------------------------------------------------------------- packing
def pack(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.uint8)
    N, K = q.shape
    out = np.empty((N, K // 8), dtype=np.int32)
    _load().oracle_pack(_ptr(q), N, K, _ptr(out))
    return out


def unpack(qweight: np.ndarray, K: int) -> np.ndarray:
    qweight = _c(qweight, np.int32)
    N = qweight.shape[0]
    out = np.empty((N, K), dtype=np.uint8)
    _load().oracle_unpack(_ptr(qweight), N, K, _ptr(out))
    return out


def pack_zeros(z: np.ndarray) -> np.ndarray:
    z = _c(z, np.uint8)
    N, ng = z.shape
    out = np.empty((N // 8, ng), dtype=np.int32)
    _load().oracle_pack_zeros(_ptr(z), N, ng, _ptr(out))
    return out


def unpack_zeros(qzeros: np.ndarray, N: int) -> np.ndarray:
    qzeros = _c(qzeros, np.int32)
    ng = qzeros.shape[1]
    out = np.empty((N, ng), dtype=np.uint8)
    _load().oracle_unpack_zeros(_ptr(qzeros), N, ng, _ptr(out))
    return out


# ---------------------------------------------------------------- dequant / gemm
def dequant(qweight, scales, qzeros, G: int, N: int, K: int, dtype: int) -> np.ndarray:
    """W_ref[n, k] = RN_dtype((q - z) * s) as uint16 bit patterns [N, K]."""
    qweight = _c(qweight, np.int32)
    scales = _c(scales, np.uint16)
    qzeros = _c(qzeros, np.int32)
    out = np.empty((N, K), dtype=np.uint16)
    _load().oracle_dequant(_ptr(qweight), _ptr(scales), _ptr(qzeros), G, N, K, dtype, _ptr(out))
    return out


def round_products(d, dtype: int) -> np.ndarray:
    """[len(d), 65536] table of RN_dtype(d_i * s) over every 16-bit pattern s."""
    d = _c(d, np.int32)
    out = np.empty((d.size, 65536), dtype=np.uint16)
    _load().oracle_round_products(_ptr(d), d.size, dtype, _ptr(out))
    return out


def gemm(x, M: int, K: int, qweight, scales, qzeros, G: int, N: int, dtype: int,
         rows=None, exact_weights: bool = False) -> np.ndarray:
    """y = x . W_ref^T in float64, [len(rows) or M, N].  x is uint16 bits [M, K]."""
    x = _c(x, np.uint16)
    qweight = _c(qweight, np.int32)
    scales = _c(scales, np.uint16)
    qzeros = _c(qzeros, np.int32)
    r = None if rows is None else _c(rows, np.int32)
    R = M if r is None else r.size
    y = np.empty((R, N), dtype=np.float64)
    _load().oracle_gemm_rows(_ptr(x), M, K, _ptr(qweight), _ptr(scales), _ptr(qzeros), G, N,
                             dtype, _ptr(r), 0 if r is None else r.size,
                             1 if exact_weights else 0, _ptr(y))
    return y


def epilogue(y, N: int, dtype: int, bias=None, silu_mul: bool = False) -> np.ndarray:
    """The fused epilogue on float64 accumulations y [R, N]: + bias (uint16
    bits [N] or None), then optionally SiLU(gate) * up over the two column
    halves.  Float64 [R, N] or [R, N / 2]."""
    y = _c(y, np.float64)
    R = y.shape[0]
    b = None if bias is None else _c(bias, np.uint16)
    out = np.empty((R, N // 2 if silu_mul else N), dtype=np.float64)
    _load().oracle_epilogue(_ptr(y), R, N, _ptr(b), dtype, 1 if silu_mul else 0, _ptr(out))
    return out


def moe_gemm(x, T: int, K: int, qweight, scales, qzeros, G: int, N: int, expert_ids, dtype: int,
             route_weights=None) -> np.ndarray:
    """Grouped skinny GEMM over routed experts, float64 [T, topk, N]:
    out[t, j] = x[t] . W_ref(e)^T with e = expert_ids[t, j], the expert's
    weight W_ref(e) = RN_dtype((q - z) * s) from qweight[e] [N, K/8],
    scales[e] [N, K/G] and qzeros[e] [N/8, K/G] (or symmetric), times
    route_weights[t, j] when given.  Each (token, expert) pair is one call of
    gemm() above on that token's row and that expert's slices."""
    x = _c(x, np.uint16).reshape(T, K)
    ids = np.asarray(expert_ids, dtype=np.int64).reshape(T, -1)
    topk = ids.shape[1]
    out = np.zeros((T, topk, N), dtype=np.float64)
    for t in range(T):
        for j in range(topk):
            e = int(ids[t, j])
            y = gemm(x[t:t + 1], 1, K, qweight[e], scales[e], None if qzeros is None else qzeros[e], G, N,
                     dtype)[0]
            if route_weights is not None:
                y = y * float(np.asarray(route_weights, dtype=np.float64).reshape(T, topk)[t, j])
            out[t, j] = y
    return out


def num_threads() -> int:
    return _load().oracle_num_threads()


# ---------------------------------------------------------------- numpy restatement
# A second, independent statement of the same definitions, used only on tiny
# inputs to cross-check the C code (brute force per group, different loops).
def np_unpack(qweight: np.ndarray, K: int) -> np.ndarray:
    words = qweight.astype(np.int64) & 0xFFFFFFFF
    shifts = 4 * np.arange(8, dtype=np.int64)
    nib = (words[:, :, None] >> shifts[None, None, :]) & 0xF
    return nib.reshape(qweight.shape[0], K).astype(np.uint8)


def np_unpack_zeros(qzeros: np.ndarray, N: int) -> np.ndarray:
    words = qzeros.astype(np.int64) & 0xFFFFFFFF            # [N/8, ng]
    shifts = 4 * np.arange(8, dtype=np.int64)
    nib = (words[:, None, :] >> shifts[None, :, None]) & 0xF  # [N/8, 8, ng]
    return nib.reshape(N, qzeros.shape[1]).astype(np.uint8)


def np_gemm_bruteforce(x_vals: np.ndarray, w_vals: np.ndarray, G: int) -> np.ndarray:
    """y[m, n] = sum over groups of (sum over k in group of x * w), plain loops."""
    M, K = x_vals.shape
    N = w_vals.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            total = 0.0
            for g in range(K // G):
                part = 0.0
                for k in range(g * G, (g + 1) * G):
                    part += float(x_vals[m, k]) * float(w_vals[n, k])
                total += part
            y[m, n] = total
    return y
