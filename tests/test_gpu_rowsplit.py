"""GPU parity of the fused prefill's row split: two launches over weight rows
[0, n_split) and [n_split, N), the second writing a column block of y with
the full output row stride, each with the configuration the dispatcher
picks for its part (with or without a K split).  Forced at chosen rows
through the test hook:

* against the oracle within the contract's tolerance, with and without
  bias, fp16 and bf16, symmetric and asymmetric, G = 32 / 64 / 128, ragged
  last row blocks;
* bit-equal to the single launch and to the oracle's rounded sum on
  integer-exact inputs (s = 1, integer x), for the fused kernel and for the
  dense form (the dequantised prefill cache).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import bits_to_tensor, check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

PREFILL = 2


def seeded_bias(N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    t = (torch.rand((N,), generator=g) * 4.0 - 2.0).to(torch.float16 if dtype == 0 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def run(w, p, d, bias_bits=None, split=None):
    bias = None if bias_bits is None else bits_to_tensor(bias_bits, p.dtype)
    if split is not None:
        w.w4a16_debug_set_config(8, [split])
    try:
        out = w.w4a16_gemm_fused(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G, bias=bias, path=PREFILL)
        torch.cuda.synchronize()
    finally:
        if split is not None:
            w.w4a16_debug_set_config(8, None)
    return out


@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("M,N,K,G,split", [(40, 776, 1024, 32, 256), (300, 1032, 512, 64, 512),
                                           (129, 1280, 768, 128, 1024)])
def test_row_split_parity(cuda_lib, M, N, K, G, split, sym, dtype, with_bias):
    w = cuda_lib
    p = make_problem(M, N, K, G, sym, dtype, seed=15000 + M + N + K + G)
    d = to_device(p, w)
    b = seeded_bias(N, dtype, seed=N + split) if with_bias else None
    out = run(w, p, d, b, split=split)
    y = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
    check_tolerance(out_values(out), oracle.epilogue(y, N, dtype, bias=b),
                    f"row split at {split}: M={M} N={N} K={K} G={G}")
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("split", [256, 512, 768])
def test_row_split_integer_exact(cuda_lib, split):
    w = cuda_lib
    M, N, K, G = 96, 1000, 1024, 64
    p = make_problem(M, N, K, G, False, 1, seed=15100 + split, x_kind="int4")
    p.scales[:] = 0x3F80                               # bf16 1.0: every partial sum is an exact integer
    d = to_device(p, w)
    single = run(w, p, d)
    parts = run(w, p, d, split=split)
    assert np.array_equal(tensor_to_bits(parts), tensor_to_bits(single))
    want = oracle.round_array(oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1), 1)
    assert np.array_equal(tensor_to_bits(parts), want)
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("split", [256, 768])
def test_dense_row_split(cuda_lib, split, with_bias):
    """The dense form (the dequantised prefill cache) split the same way:
    bit-equal to its single launch and to the oracle's rounded sum on
    integer-exact data, with and without bias."""
    w = cuda_lib
    M, N, K, G = 72, 1000, 1024, 128
    p = make_problem(M, N, K, G, True, 1, seed=15200 + split, x_kind="int4")
    p.scales[:] = 0x3F80
    d = to_device(p, w)
    cache = w.w4a16_dequantize(d["qweight"], d["scales"], d["qzeros"], G)
    g = torch.Generator().manual_seed(split)
    bias_t = torch.randint(-8, 9, (N,), generator=g).to(torch.bfloat16).cuda() if with_bias else None
    single = w.w4a16_gemm_dense(d["x"], cache, bias=bias_t)
    w.w4a16_debug_set_config(8, [split])
    try:
        parts = w.w4a16_gemm_dense(d["x"], cache, bias=bias_t)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(8, None)
    assert np.array_equal(tensor_to_bits(parts), tensor_to_bits(single))
    y = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1)
    bb = tensor_to_bits(bias_t) if with_bias else None
    assert np.array_equal(tensor_to_bits(parts), oracle.round_array(oracle.epilogue(y, N, 1, bias=bb), 1))
    assert w.w4a16_last_device_error() == 0
