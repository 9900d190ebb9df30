"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

* packing and dequantisation: bit-exact;
* GEMM: |y - y_ref| <= 1e-2 max(1, |y_ref|) elementwise and relative L2
  <= 5e-3, on shapes spanning several tiles with ragged tails, every group
  size, symmetric and asymmetric weights, fp16 and bf16, both kernels;
* integer-exact GEMM (s = 1, integer x): bit-exact outputs, which catches any
  layout, swizzle or split-K indexing error with zero tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from golden_cases import load, to_bits
from parity_helpers import (bits_to_tensor, check_tolerance, out_values, tensor_to_bits,
                            to_device)
from w4a16_group_quantised_gb300.workloads import make_problem, tiny_symmetric

pytestmark = pytest.mark.gpu

DECODE, PREFILL = 1, 2


def run_case(w, p, path, rows=None):
    d = to_device(p, w)
    out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G, path=path)
    torch.cuda.synchronize()
    y = out_values(out)
    y_ref = oracle.gemm(p.x, p.M, p.K, d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, p.dtype,
                        rows=rows)
    if rows is not None:
        y = y[rows]
    check_tolerance(y, y_ref, f"M={p.M} N={p.N} K={p.K} G={p.G} sym={p.sym} dt={p.dtype} path={path}")
    return y, y_ref


# ------------------------------------------------------------------ packing / dequant
ROUTINES = [0, 1, 2]          # prefill, decode (runtime constants), balanced decode
ROUTINE_IDS = ["prefill", "decode", "balanced"]


@pytest.mark.parametrize("routine", ROUTINES, ids=ROUTINE_IDS)
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("G", [32, 64, 128])
def test_dequant_bit_exact(cuda_lib, dtype, sym, G, routine):
    """Each GEMM kernel's own dequantiser, run over a whole matrix and written
    in natural order, equals the oracle's RN((q - z) * s) bit for bit."""
    w = cuda_lib
    p = make_problem(1, 264, 1152, G, sym, dtype, seed=100 + G)
    d = to_device(p, w)
    got = tensor_to_bits(w.w4a16_dequant_debug(d["qweight"], d["scales"], d["qzeros"], G,
                                               routine=routine))
    ref = oracle.dequant(d["ref_qw"], p.scales, d["ref_qz"], G, p.N, p.K, dtype)
    assert np.array_equal(got, ref)


def exhaustive_case(dtype):
    """Row n holds scale bit pattern n (non-finite patterns replaced by 0);
    group 0 has z = 15 (q - z = -15..0), group 1 z = 0 (q - z = 0..15), and
    each group runs q over 0..15 twice."""
    N, K, G = 65536, 64, 32
    pat = np.arange(65536, dtype=np.uint16)
    vals = oracle.bits_to_float64(pat, dtype)
    s_bits = np.where(np.isfinite(vals), pat, 0).astype(np.uint16)
    scales = np.repeat(s_bits[:, None], 2, axis=1)
    q = np.tile(np.concatenate([np.arange(16)] * 4).astype(np.uint8), (N, 1))
    z = np.tile(np.array([15, 0], dtype=np.uint8), (N, 1))
    qw = oracle.pack(q)
    qz = oracle.pack_zeros(z)
    ref = oracle.dequant(qw, scales, qz, G, N, K, dtype)
    return N, K, G, qw, qz, scales, s_bits, ref


@pytest.mark.parametrize("routine", ROUTINES, ids=ROUTINE_IDS)
@pytest.mark.parametrize("dtype", [0, 1])
def test_dequant_exhaustive_scales(cuda_lib, dtype, routine):
    """Every finite 16-bit scale pattern (normal, subnormal, zero, negative)
    times every q - z in [-15, 15], through each GEMM kernel's dequantiser:
    bit-exact against the oracle's RN_dtype((q - z) * s)."""
    w = cuda_lib
    N, K, G, qw, qz, scales, s_bits, ref = exhaustive_case(dtype)
    got = tensor_to_bits(w.w4a16_dequant_debug(torch.from_numpy(qw).cuda(),
                                               bits_to_tensor(scales, dtype),
                                               torch.from_numpy(qz).cuda(), G,
                                               routine=routine))
    sv = np.abs(oracle.bits_to_float64(s_bits, dtype))
    min_normal = 2.0 ** -14 if dtype == 0 else 2.0 ** -126
    subnormal = (sv < min_normal) & (sv > 0)
    mism = (got != ref).any(axis=1)
    assert not mism[~subnormal].any(), f"{mism[~subnormal].sum()} rows with normal scales differ"
    assert not mism[subnormal].any(), f"{mism[subnormal].sum()} rows with subnormal scales differ"


def test_pack_edge_values(cuda_lib):
    w = cuda_lib
    q = np.full((8, 32), 15, dtype=np.uint8)
    q[:, ::2] = 0
    p = torch.from_numpy(q).cuda()
    assert np.array_equal(w.w4a16_pack(p).cpu().numpy(), oracle.pack(q))
    z = np.random.default_rng(0).integers(0, 16, (64, 3), dtype=np.uint8)
    assert np.array_equal(w.w4a16_pack_zeros(torch.from_numpy(z).cuda()).cpu().numpy(),
                          oracle.pack_zeros(z))


# ------------------------------------------------------------------ hand-worked case
def test_golden_library_case(cuda_lib):
    w = cuda_lib
    c = load("lib_sym_fp16_m2_k32_n8")
    qw = torch.from_numpy(oracle.pack(c["q"])).cuda()
    x = bits_to_tensor(to_bits(c["x_vals"], 0), 0)
    s = bits_to_tensor(to_bits(c["scales_vals"], 0), 0)
    for path in (DECODE, PREFILL):
        out = out_values(w.w4a16_gemm(x, qw, s, None, 32, path=path))
        assert np.array_equal(out, c["y"]), (path, out)


# ------------------------------------------------------------------ GEMM tolerance
SMALL_SHAPES = [(8, 32), (136, 96), (264, 288), (520, 1184)]


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
def test_decode_small(cuda_lib, M, dtype, sym):
    for i, (N, K) in enumerate(SMALL_SHAPES):
        for G in (32, 64, 128):
            if K % G:
                continue
            p = make_problem(M, N, K, G, sym, dtype, seed=1000 + 10 * i + G + M)
            run_case(cuda_lib, p, DECODE)


@pytest.mark.parametrize("M", [1, 9, 16, 100, 129, 300])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
def test_prefill_small(cuda_lib, M, dtype, sym):
    for i, (N, K) in enumerate(SMALL_SHAPES):
        for G in (32, 64, 128):
            if K % G:
                continue
            p = make_problem(M, N, K, G, sym, dtype, seed=2000 + 10 * i + G + M)
            run_case(cuda_lib, p, PREFILL)


@pytest.mark.parametrize("path", [DECODE, PREFILL])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
def test_integer_exact(cuda_lib, path, dtype, sym):
    """s = 1, x integer in [-4, 4]: every fp32 partial sum is an exact
    integer, so out must equal RN_dtype(y_ref) bit for bit."""
    w = cuda_lib
    M = 5 if path == DECODE else 200
    for (N, K, G) in [(136, 288, 32), (392, 1088, 64), (264, 2560, 128)]:
        p = make_problem(M, N, K, G, sym, dtype, seed=77 + N, x_kind="int4")
        one = 0x3C00 if dtype == 0 else 0x3F80
        p.scales[:] = one
        d = to_device(p, w)
        out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=path)
        got = tensor_to_bits(out)
        y_ref = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
        assert np.all(y_ref == np.round(y_ref))
        assert np.array_equal(got, oracle.round_array(y_ref, dtype)), (N, K, G)


def test_tiny_symmetric_config(cuda_lib):
    for M in (1, 4):
        p = tiny_symmetric(M)
        run_case(cuda_lib, p, 0)
        run_case(cuda_lib, p, DECODE)
        run_case(cuda_lib, p, PREFILL)


def test_m_zero_is_noop(cuda_lib):
    w = cuda_lib
    p = make_problem(1, 64, 128, 32, True, 0, seed=3)
    d = to_device(p, w)
    out = torch.full((1, 64), 7.0, dtype=torch.float16, device="cuda")
    x0 = d["x"][:0]
    w.w4a16_gemm(x0, d["qweight"], d["scales"], None, 32, out=out[:0])
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_auto_dispatch_matches_forced(cuda_lib):
    w = cuda_lib
    for M in (1, 8, 9, 64):
        p = make_problem(M, 264, 512, 64, False, 1, seed=500 + M)
        d = to_device(p, w)
        auto = tensor_to_bits(w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 64))
        path = w.w4a16_select_path(M, 264, 512, 64, False, 1)
        forced = tensor_to_bits(w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 64,
                                             path=path))
        assert np.array_equal(auto, forced)


def test_deterministic(cuda_lib):
    w = cuda_lib
    for path, M in ((DECODE, 3), (PREFILL, 77)):
        p = make_problem(M, 1032, 4096, 128, False, 1, seed=9)
        d = to_device(p, w)
        a = tensor_to_bits(w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 128, path=path))
        b = tensor_to_bits(w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 128, path=path))
        assert np.array_equal(a, b)


def test_host_buffer_entry_point(cuda_lib):
    w = cuda_lib
    p = make_problem(3, 136, 288, 32, False, 0, seed=12)
    d = to_device(p, w)
    x_host = d["x"].cpu().pin_memory()
    out_host = torch.empty((3, 136), dtype=torch.float16).pin_memory()
    dev_x = torch.empty_like(d["x"])
    dev_out = torch.empty((3, 136), dtype=torch.float16, device="cuda")
    w.w4a16_gemm_host(x_host, d["qweight"], d["scales"], d["qzeros"], 32, out_host, dev_x, dev_out)
    ref = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 32)
    assert torch.equal(out_host, ref.cpu())


def test_host_buffer_async_entry_point(cuda_lib):
    """Several layers enqueued through w4a16_gemm_host_async on one stream,
    one synchronisation: every host result equals the device-buffer call."""
    w = cuda_lib
    stream = torch.cuda.Stream()
    cases = [make_problem(M, N, 512, 64, sym, 1, seed=20 + M) for (M, N, sym) in ((1, 264, True), (4, 520, False),
                                                                                   (40, 256, True))]
    devs = [to_device(p, w) for p in cases]
    xs = [d["x"].cpu().pin_memory() for d in devs]
    outs = [torch.full((p.M, p.N), 7.0, dtype=torch.bfloat16).pin_memory() for p in cases]
    dxs = [torch.empty_like(d["x"]) for d in devs]
    dos = [torch.empty((p.M, p.N), dtype=torch.bfloat16, device="cuda") for p in cases]
    torch.cuda.synchronize()
    for p, d, x, o, a, b in zip(cases, devs, xs, outs, dxs, dos):
        w.w4a16_gemm_host_async(x, d["qweight"], d["scales"], d["qzeros"], p.G, o, a, b, stream=stream)
    stream.synchronize()
    for p, d, o in zip(cases, devs, outs):
        ref = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G)
        torch.cuda.synchronize()
        assert torch.equal(o, ref.cpu())


def test_device_status_clean(cuda_lib):
    torch.cuda.synchronize()
    assert cuda_lib.w4a16_last_device_error() == 0


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
def test_prefill_k_split_integer_exact(cuda_lib, dtype, sym):
    """Few output tiles: the prefill kernel splits K over a cluster of 2 to 8
    CTAs (whole 256-k weight tiles each, uneven shares, a ragged K tail in
    the last one) and sums the partial tiles across the cluster.  s = 1 and
    integer x make every partial sum exact: bit-exact outputs, twice in a row."""
    w = cuda_lib
    cases = [(16, 256, 512, 32), (37, 200, 768, 64), (100, 256, 1184, 32),
             (64, 512, 2560, 128), (129, 1000, 4096, 128), (48, 2056, 1344, 64)]
    for (M, N, K, G) in cases:
        p = make_problem(M, N, K, G, sym, dtype, seed=900 + M + N, x_kind="int4")
        p.scales[:] = 0x3C00 if dtype == 0 else 0x3F80
        d = to_device(p, w)
        y_ref = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
        want = oracle.round_array(y_ref, dtype)
        for _ in range(2):
            out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=PREFILL)
            assert np.array_equal(tensor_to_bits(out), want), (M, N, K, G)
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("ks", [1, 2, 4, 7, 8])
def test_prefill_forced_k_split(cuda_lib, ks):
    """Every cluster size gives the same bit-exact integer result (nine 256-k
    weight tiles: shares of one to five tiles; ragged M and N)."""
    w = cuda_lib
    M, N, K, G = 61, 520, 2304, 64
    p = make_problem(M, N, K, G, False, 1, seed=4242, x_kind="int4")
    p.scales[:] = 0x3F80
    d = to_device(p, w)
    want = oracle.round_array(oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1), 1)
    w.w4a16_debug_set_config(2, [64, 4, 2, 2, ks])
    try:
        out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=PREFILL)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(2, None)
    assert np.array_equal(tensor_to_bits(out), want)
    assert w.w4a16_last_device_error() == 0


DECODE_FORCED = [[1, 4, 4, 2, 5], [1, 8, 2, 3, 2], [2, 4, 2, 2, 3], [1, 4, 4, 4, 8], [1, 2, 4, 3, 7], [2, 8, 1, 2, 2]]


@pytest.mark.parametrize("cfg", DECODE_FORCED, ids=lambda c: "-".join(map(str, c)))
@pytest.mark.parametrize("sym", [True, False])
def test_decode_forced_config_integer_exact(cuda_lib, cfg, sym):
    """Every decode configuration family, forced through the tuning hook,
    gives the oracle's result bit for bit on integer-exact inputs (ragged N
    and K tails, cluster sizes 1 to 8, one or two row blocks per warp, one to
    four boxes per stage, M up to 8)."""
    w = cuda_lib
    for (M, N, K, G) in [(1, 264, 2560, 128), (3, 1000, 1184, 32), (8, 520, 4096, 64)]:
        p = make_problem(M, N, K, G, sym, 1, seed=7100 + M + N, x_kind="int4")
        p.scales[:] = 0x3F80
        d = to_device(p, w)
        want = oracle.round_array(oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1), 1)
        w.w4a16_debug_set_config(1, cfg)
        try:
            out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=DECODE)
            torch.cuda.synchronize()
        finally:
            w.w4a16_debug_set_config(1, None)
        assert np.array_equal(tensor_to_bits(out), want), (cfg, M, N, K, G)
    assert w.w4a16_last_device_error() == 0
