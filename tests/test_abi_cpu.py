"""Host-side checks that need no GPU: the library builds for sm_103a, loads,
exports every entry point include/w4a16.h declares, and rejects invalid
arguments on the host before touching the device; the dispatcher is host
logic."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    from w4a16_group_quantised_gb300 import build
    build.build()
    import w4a16_group_quantised_gb300 as w
    return w.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\bint\s+(w4a16_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("w4a16_pack", "w4a16_pack_zeros", "w4a16_dequant_debug", "w4a16_gemm"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.w4a16_version() == 100


NULL = None
ALIGNED = ctypes.c_void_p(0x1000)     # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x1008)
ODD = ctypes.c_void_p(0x1001)


def gemm(lib, x=ALIGNED, M=1, K=128, qw=ALIGNED, s=ALIGNED, qz=NULL, G=32, N=64, out=ALIGNED,
         dtype=0):
    return lib.w4a16_gemm(x, M, K, qw, s, qz, G, N, out, None, dtype)


def test_validation_codes(lib):
    assert gemm(lib, G=48) == -3                # W4A16_ERR_GROUP
    assert gemm(lib, G=16) == -3
    assert gemm(lib, K=96, G=64) == -3          # K % G
    assert gemm(lib, N=60) == -2                # W4A16_ERR_SHAPE: N % 8
    assert gemm(lib, M=-1) == -2
    assert gemm(lib, K=0) == -2
    assert gemm(lib, dtype=2) == -5             # W4A16_ERR_DTYPE
    assert gemm(lib, qw=NULL) == -1             # W4A16_ERR_NULL
    assert gemm(lib, s=NULL) == -1
    assert gemm(lib, x=NULL) == -1
    assert gemm(lib, out=NULL) == -1
    assert gemm(lib, x=MISALIGNED) == -4        # W4A16_ERR_ALIGN
    assert gemm(lib, qz=MISALIGNED) == -4
    assert gemm(lib, N=1 << 20, K=1 << 15) == -2   # int32 index headroom
    # M == 0 is a valid no-op: nothing is launched, no device needed
    assert gemm(lib, M=0, x=NULL, out=NULL) == 0


def test_forced_path_limits(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    ex = lib.w4a16_gemm_ex
    assert ex(ALIGNED, 9, 128, ALIGNED, ALIGNED, None, 32, 64, ALIGNED, None, 0, 1) == -2
    assert ex(ALIGNED, 1, 128, ALIGNED, ALIGNED, None, 32, 64, ALIGNED, None, 0, 7) == -9
    assert ex(ALIGNED, 0, 128, ALIGNED, ALIGNED, None, 32, 64, ALIGNED, None, 0, 2) == 0


def test_noalloc_entry_point_limits(lib):
    """The allocation-free decode entry point validates on the host like
    w4a16_gemm and rejects what its static scratch cannot hold."""
    f = lib.w4a16_gemm_decode_noalloc
    assert f(ALIGNED, 9, 128, ALIGNED, ALIGNED, None, 32, 64, ALIGNED, None, 0) == -2     # M > 8
    assert f(ALIGNED, 1, 128, ALIGNED, ALIGNED, None, 32, 131080, ALIGNED, None, 0) == -2  # N > 131072
    assert f(ALIGNED, 1, 128, ALIGNED, ALIGNED, None, 48, 64, ALIGNED, None, 0) == -3     # group size
    assert f(MISALIGNED, 1, 128, ALIGNED, ALIGNED, None, 32, 64, ALIGNED, None, 0) == -4
    assert f(None, 0, 128, ALIGNED, ALIGNED, None, 32, 64, None, None, 0) == 0            # M == 0
    # staged x (M x K) plus the partial slots must fit in the kernel's shared memory
    assert f(ALIGNED, 8, 14336, ALIGNED, ALIGNED, None, 128, 4096, ALIGNED, None, 0) == -2


def test_pack_validation(lib):
    assert lib.w4a16_pack(ALIGNED, 8, 12, ALIGNED, None) == -2     # K % 8
    assert lib.w4a16_pack(NULL, 8, 16, ALIGNED, None) == -1
    assert lib.w4a16_pack(MISALIGNED, 8, 16, ALIGNED, None) == -4
    assert lib.w4a16_pack(NULL, 0, 16, NULL, None) == 0            # empty is a no-op
    assert lib.w4a16_pack_zeros(ALIGNED, 12, 4, ALIGNED, None) == -2  # N % 8
    assert lib.w4a16_pack_zeros(NULL, 0, 4, NULL, None) == 0


def test_dequant_validation(lib):
    f = lib.w4a16_dequant_debug
    assert f(ALIGNED, ALIGNED, None, 40, 64, 160, ALIGNED, 0, None) == -3
    assert f(ALIGNED, ALIGNED, None, 32, 63, 128, ALIGNED, 0, None) == -2
    assert f(NULL, ALIGNED, None, 32, 64, 128, ALIGNED, 0, None) == -1
    assert f(ALIGNED, ALIGNED, None, 32, 64, 128, ALIGNED, 3, None) == -5


def test_dispatcher_is_host_logic(lib):
    assert lib.w4a16_select_path(1, 4096, 4096, 128, 1, 1) == 1     # decode
    assert lib.w4a16_select_path(8, 4096, 4096, 128, 0, 0) == 1
    assert lib.w4a16_select_path(1920, 4096, 4096, 64, 0, 1) == 2   # prefill
    assert lib.w4a16_select_path(1, 4096, 4096, 48, 1, 1) == -3
    for M in (1, 2, 3, 4, 5, 6, 8, 16, 32, 64, 128, 4096):
        r = lib.w4a16_select_path(M, 2560, 9728, 128, 1, 0)
        assert r in (1, 2)
        if M > 8:
            assert r == 2


def test_debug_config_validation(lib):
    arr = (ctypes.c_int * 4)(24, 3, 2, 2)
    assert lib.w4a16_debug_set_config(2, arr, 4) == -9   # BN not a multiple of 16
    arr = (ctypes.c_int * 4)(256, 8, 2, 2)
    assert lib.w4a16_debug_set_config(2, arr, 4) == -9   # rings do not fit in shared memory
    arr = (ctypes.c_int * 4)(128, 3, 2, 2)
    assert lib.w4a16_debug_set_config(2, arr, 4) == 0
    arr = (ctypes.c_int * 5)(128, 3, 2, 2, 8)
    assert lib.w4a16_debug_set_config(2, arr, 5) == 0    # K split over 8 CTAs
    arr = (ctypes.c_int * 5)(128, 3, 2, 2, 9)
    assert lib.w4a16_debug_set_config(2, arr, 5) == -9   # more than 8 CTAs
    arr = (ctypes.c_int * 5)(256, 3, 2, 2, 2)
    assert lib.w4a16_debug_set_config(2, arr, 5) == -9   # 256 KB partial tile does not fit
    arr = (ctypes.c_int * 4)(256, 3, 3, 2)
    assert lib.w4a16_debug_set_config(2, arr, 4) == 0    # fits the dense form (no packed ring) only
    arr = (ctypes.c_int * 6)(128, 4, 3, 2, 1, 1)
    assert lib.w4a16_debug_set_config(2, arr, 6) == 0    # swapped operands at BN = 128
    arr = (ctypes.c_int * 6)(256, 2, 3, 2, 1, 1)
    assert lib.w4a16_debug_set_config(2, arr, 6) == -9   # swapped operands need BN = 128
    arr = (ctypes.c_int * 6)(128, 4, 3, 2, 1, 2)
    assert lib.w4a16_debug_set_config(2, arr, 6) == -9   # swap flag is 0 or 1
    for bad in (0, -256, 100):                            # row split: a positive multiple of 256
        arr = (ctypes.c_int * 1)(bad)
        assert lib.w4a16_debug_set_config(8, arr, 1) == -9
    arr = (ctypes.c_int * 1)(512)
    assert lib.w4a16_debug_set_config(8, arr, 1) == 0
    assert lib.w4a16_debug_set_config(8, None, 0) == 0
    assert lib.w4a16_debug_set_config(2, None, 0) == 0
    assert lib.w4a16_debug_set_config(9, None, 0) == -9
    assert lib.w4a16_debug_set_config(5, None, 0) == -9   # no such hook
    assert lib.w4a16_debug_set_config(6, None, 0) == -9
    assert lib.w4a16_debug_set_config(7, None, 0) == 0    # timeout-path test hook off
    arr = (ctypes.c_int * 2)(1, 1)
    assert lib.w4a16_debug_set_config(7, arr, 2) == -9


def test_fused_entry_point_limits(lib):
    """w4a16_gemm_fused: host validation of the epilogue and bias arguments."""
    f = lib.w4a16_gemm_fused
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    args = lambda M=1, bias=None, epi=0, path=0: f(ALIGNED, M, 128, ALIGNED, ALIGNED, None, 32, 64, bias, epi,
                                                  ALIGNED, None, 0, path)
    assert args(epi=2) == -9                       # unknown epilogue
    assert args(epi=1, M=9) == -2                  # SiLU-and-multiply is a decode epilogue
    assert args(epi=1, path=2) == -9               # ... not on the prefill kernel
    assert args(bias=ODD) == -4                    # bias must be 2-byte aligned
    assert args(M=0, epi=1) == 0                   # empty is a no-op
    assert args(M=0, bias=ALIGNED) == 0


def _cpu(*shape, dtype=None):
    import torch
    return torch.zeros(*shape, dtype=dtype or torch.float16)


def test_binding_rejects_wrong_zero_point_dtype():
    """The packed zero-point contract: int32 only (a float tensor of zero
    points is refused before the library is called)."""
    import torch
    from w4a16_group_quantised_gb300 import binding as b
    with pytest.raises(TypeError):
        b._check_gemm_operands(_cpu(1, 64), _cpu(8, 8, dtype=torch.int32), _cpu(8, 2), _cpu(1, 2), 32, None,
                               require_cuda=False)


def test_binding_operand_checks():
    """Types, dtypes, shapes, layout and device are checked before the C
    call: TypeError for a type or dtype, ValueError for the rest."""
    import torch
    from w4a16_group_quantised_gb300 import binding as b
    i32 = torch.int32
    x, qw, s, qz = _cpu(2, 64), _cpu(16, 8, dtype=i32), _cpu(16, 2), _cpu(2, 2, dtype=i32)
    ok = dict(require_cuda=False)
    assert b._check_gemm_operands(x, qw, s, qz, 32, _cpu(2, 16), **ok) == (2, 64, 16)
    with pytest.raises(ValueError, match="CUDA"):
        b._check_gemm_operands(x, qw, s, qz, 32, None)                       # CPU tensors
    with pytest.raises(TypeError):
        b._check_gemm_operands(x.float(), qw, s, qz, 32, None, **ok)          # fp32 activations
    with pytest.raises(TypeError):
        b._check_gemm_operands(x, qw.to(torch.int64), s, qz, 32, None, **ok)  # int64 weights
    with pytest.raises(TypeError):
        b._check_gemm_operands(x, qw, s.to(torch.bfloat16), qz, 32, None, **ok)   # scales dtype
    with pytest.raises(TypeError):
        b._check_gemm_operands(x, qw, s, qz, 32.0, None, **ok)                 # G not an int
    with pytest.raises(TypeError):
        b._check_gemm_operands(x.numpy(), qw, s, qz, 32, None, **ok)           # not a tensor
    with pytest.raises(ValueError, match="contiguous"):
        b._check_gemm_operands(_cpu(64, 2).t(), qw, s, qz, 32, None, **ok)
    with pytest.raises(ValueError, match="qweight"):
        b._check_gemm_operands(x, _cpu(16, 4, dtype=i32), s, qz, 32, None, **ok)
    with pytest.raises(ValueError, match="scales"):
        b._check_gemm_operands(x, qw, _cpu(16, 4), qz, 32, None, **ok)
    with pytest.raises(ValueError, match="qzeros"):
        b._check_gemm_operands(x, qw, s, _cpu(16, 2, dtype=i32), 32, None, **ok)
    with pytest.raises(ValueError, match="out"):
        b._check_gemm_operands(x, qw, s, qz, 32, _cpu(2, 8), **ok)
    with pytest.raises(TypeError):
        b._check_gemm_operands(x, qw, s, qz, 32, _cpu(2, 16, dtype=torch.bfloat16), **ok)
    with pytest.raises(ValueError, match="bias"):
        b._check_gemm_operands(x, qw, s, qz, 32, None, bias=_cpu(8), **ok)
    # SiLU-and-multiply writes [M, N/2]
    assert b._check_gemm_operands(x, qw, s, None, 32, _cpu(2, 8), out_cols=8, **ok) == (2, 64, 16)


class _Layer(ctypes.Structure):
    _fields_ = [("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("qzeros_or_null", ctypes.c_void_p), ("bias_or_null", ctypes.c_void_p),
                ("G", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("epilogue", ctypes.c_int), ("out", ctypes.c_void_p)]


def test_chain_entry_point_limits(lib):
    """w4a16_gemm_chain checks the whole chain on the host first: widths must
    chain (a SiLU-and-multiply layer halves its width), layers non-null."""
    f = lib.w4a16_gemm_chain
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    a = ALIGNED.value

    def layers(*specs):
        arr = (_Layer * len(specs))(*[_Layer(a, a, None, None, 32, N, K, epi, a) for (N, K, epi) in specs])
        return ctypes.cast(arr, ctypes.c_void_p), arr

    p, keep = layers((64, 128, 0), (32, 64, 0))
    assert f(ALIGNED, 0, p, 2, 0, None) == 0                   # M == 0: nothing to do
    p, keep = layers((64, 128, 0), (32, 96, 0))
    assert f(ALIGNED, 1, p, 2, 0, None) == -2                  # 96 != 64
    p, keep = layers((64, 128, 1), (32, 64, 0))
    assert f(ALIGNED, 1, p, 2, 0, None) == -2                  # SiLU halves 64 -> 32
    p, keep = layers((64, 128, 3))
    assert f(ALIGNED, 1, p, 1, 0, None) == -9                  # unknown epilogue
    p, keep = layers((64, 128, 1))
    assert f(ALIGNED, 9, p, 1, 0, None) == -2                  # SiLU needs M <= 8
    assert f(ALIGNED, 1, None, 2, 0, None) == -1
    assert f(ALIGNED, 1, None, 0, 0, None) == 0
    assert f(ALIGNED, 1, None, -1, 0, None) == -9


def test_cache_entry_point_limits(lib):
    """w4a16_gemm_dense / w4a16_dequantize / w4a16_gemm_cached validate on the host."""
    f = lib.w4a16_gemm_dense
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert f(ALIGNED, 1, 100, ALIGNED, 64, None, ALIGNED, 0, None) == -2      # K % 8
    assert f(ALIGNED, 1, 128, ALIGNED, 60, None, ALIGNED, 0, None) == -2      # N % 8
    assert f(ALIGNED, 1, 128, NULL, 64, None, ALIGNED, 0, None) == -1
    assert f(MISALIGNED, 1, 128, ALIGNED, 64, None, ALIGNED, 0, None) == -4
    assert f(ALIGNED, 1, 128, ALIGNED, 64, ODD, ALIGNED, 0, None) == -4
    assert f(ALIGNED, 1, 128, ALIGNED, 64, None, ALIGNED, 5, None) == -5
    assert f(None, 0, 128, ALIGNED, 64, None, None, 0, None) == 0             # M == 0
    g = lib.w4a16_dequantize
    g.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert g(ALIGNED, ALIGNED, None, 40, 64, 160, ALIGNED, 0, None) == -3
    h = lib.w4a16_gemm_cached
    h.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + \
        [ctypes.c_void_p] * 3 + [ctypes.c_int]
    assert h(ALIGNED, 1, 128, ALIGNED, ALIGNED, None, 48, 64, ALIGNED, ALIGNED, None, 0) == -3
    assert h(None, 0, 128, ALIGNED, ALIGNED, None, 32, 64, ALIGNED, None, None, 0) == 0


def test_moe_entry_point_limits(lib):
    f = lib.w4a16_moe_gemm
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, I, I, P, P, P, I, I, I, P, I, P, P, I, P]
    call = lambda T=1, K=128, G=32, N=64, E=4, ids=ALIGNED, topk=2, rw=None, x=ALIGNED: f(
        x, T, K, ALIGNED, ALIGNED, None, G, N, E, ids, topk, rw, ALIGNED, 0, None)
    assert call(E=0) == -2
    assert call(topk=0) == -2
    assert call(T=-1) == -2
    assert call(N=60) == -2
    assert call(G=48) == -3
    assert call(ids=None) == -1
    assert call(rw=ctypes.c_void_p(0x1002)) == -4
    assert call(x=MISALIGNED) == -4
    assert call(T=0, ids=None, x=None) == 0
