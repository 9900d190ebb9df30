"""GPU parity of the dequantised prefill cache: w4a16_dequantize builds
W = RN((q - z) s) bit for bit; w4a16_gemm_dense multiplies by it on the
tensor cores (weights loaded by TMA, no dequantisation) within the contract's
tolerance, bit-exact on integer-exact inputs, with ragged M, N and K tails,
bias, and forced K splits; w4a16_gemm_cached routes decode-sized M to the
int4 kernel and prefill-sized M to the cache."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import bits_to_tensor, check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import llama31_8b_prefill, make_problem

pytestmark = pytest.mark.gpu


def cache_of(w, p, d):
    wc = w.w4a16_dequantize(d["qweight"], d["scales"], d["qzeros"], p.G)
    torch.cuda.synchronize()
    ref = oracle.dequant(d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, p.K, p.dtype)
    assert np.array_equal(tensor_to_bits(wc), ref), "dequantised cache differs from the oracle"
    return wc


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("M,N,K,G,sym", [(9, 264, 1152, 128, True), (200, 1000, 1184, 32, False),
                                         (1, 520, 4096, 64, False), (333, 2048, 2560, 128, True),
                                         (64, 8, 64, 32, False)])
def test_dense_gemm(cuda_lib, M, N, K, G, sym, dtype):
    w = cuda_lib
    p = make_problem(M, N, K, G, sym, dtype, seed=14000 + M + N)
    d = to_device(p, w)
    wc = cache_of(w, p, d)
    out = w.w4a16_gemm_dense(d["x"], wc)
    torch.cuda.synchronize()
    ref = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
    check_tolerance(out_values(out), ref, f"dense M={M} N={N} K={K}")
    g = torch.Generator().manual_seed(M)
    bias = (torch.rand((N,), generator=g) - 0.5).to(d["x"].dtype).cuda()
    out = w.w4a16_gemm_dense(d["x"], wc, bias=bias)
    torch.cuda.synchronize()
    bb = tensor_to_bits(bias)
    check_tolerance(out_values(out), oracle.epilogue(ref, N, dtype, bias=bb), f"dense+bias M={M} N={N} K={K}")
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("ks", [1, 2, 4, 8])
def test_dense_integer_exact_k_split(cuda_lib, ks):
    w = cuda_lib
    M, N, K, G = 96, 520, 4096, 128
    p = make_problem(M, N, K, G, False, 1, seed=14100 + ks, x_kind="int4")
    p.scales[:] = 0x3F80
    d = to_device(p, w)
    wc = cache_of(w, p, d)
    w.w4a16_debug_set_config(2, [96, 3, 3, 2, ks])
    try:
        out = w.w4a16_gemm_dense(d["x"], wc)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(2, None)
    want = oracle.round_array(oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1), 1)
    assert np.array_equal(tensor_to_bits(out), want)
    assert w.w4a16_last_device_error() == 0


def test_dense_only_override(cuda_lib):
    """A forced configuration that fits the dense form only (no room left
    for the packed-weight ring) runs the dense GEMM, bit-exact on integer
    data, and the fused GEMM refuses it with W4A16_ERR_ARG."""
    w = cuda_lib
    M, N, K, G = 256, 512, 2048, 128
    p = make_problem(M, N, K, G, False, 1, seed=14300, x_kind="int4")
    p.scales[:] = 0x3F80
    d = to_device(p, w)
    wc = cache_of(w, p, d)
    w.w4a16_debug_set_config(2, [256, 3, 3, 2])
    try:
        out = w.w4a16_gemm_dense(d["x"], wc)
        torch.cuda.synchronize()
        with pytest.raises(w.W4A16Error) as ei:
            w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G)
        assert ei.value.code == -9
    finally:
        w.w4a16_debug_set_config(2, None)
    want = oracle.round_array(oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1), 1)
    assert np.array_equal(tensor_to_bits(out), want)
    assert w.w4a16_last_device_error() == 0


def test_cached_routing(cuda_lib):
    """Decode-sized M reads int4 (same bits as w4a16_gemm); prefill-sized M
    reads the cache (same bits as w4a16_gemm_dense)."""
    w = cuda_lib
    p = make_problem(64, 1024, 2048, 128, False, 1, seed=14200)
    d = to_device(p, w)
    wc = cache_of(w, p, d)
    for M in (1, 8, 9, 64):
        x = d["x"][:M]
        got = w.w4a16_gemm_cached(x, d["qweight"], d["scales"], d["qzeros"], p.G, w_cache=wc)
        if M <= 8:
            want = w.w4a16_gemm(x, d["qweight"], d["scales"], d["qzeros"], p.G)
        else:
            want = w.w4a16_gemm_dense(x, wc)
        torch.cuda.synchronize()
        assert torch.equal(got, want), M
        nocache = w.w4a16_gemm_cached(x, d["qweight"], d["scales"], d["qzeros"], p.G)
        assert torch.equal(nocache, w.w4a16_gemm(x, d["qweight"], d["scales"], d["qzeros"], p.G)), M


@pytest.mark.parametrize("shape", range(4))
def test_dense_fullsize_llama_prefill(cuda_lib, shape):
    """The Llama-3.1-8B-shaped layers at M = 1920 through the cache: sampled
    rows (first, last, 14 seeded) against the oracle."""
    w = cuda_lib
    p = llama31_8b_prefill(shape, 1920)
    d = to_device(p, w)
    wc = cache_of(w, p, d)
    out = w.w4a16_gemm_dense(d["x"], wc)
    torch.cuda.synchronize()
    rng = np.random.default_rng(shape)
    rows = np.unique(np.concatenate([[0, 1919], rng.integers(0, 1920, 14)])).astype(np.int32)
    ref = oracle.gemm(p.x, p.M, p.K, d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, p.dtype, rows=rows)
    check_tolerance(out_values(out)[rows], ref, f"dense llama shape {shape}")
    assert w.w4a16_last_device_error() == 0
