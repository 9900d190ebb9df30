"""GPU parity of the prefill kernel's swapped form (x as the MMA's A operand,
128 tokens; the tile's 256 dequantised weight rows as B, N = 256), forced
through the tuning hook:

* against the oracle within the contract's tolerance, with and without a K
  split over a cluster, with and without bias, fp16 and bf16, symmetric and
  asymmetric, M not a multiple of 128, N not a multiple of 256;
* bit-equal to the plain form and to the oracle's rounded sum on
  integer-exact inputs (s = 1, integer x), for the fused kernel and the
  dense form.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import bits_to_tensor, check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

PREFILL = 2


def forced(w, cfg, fn):
    w.w4a16_debug_set_config(2, cfg)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(2, None)
    return out


def seeded_bias(N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    t = (torch.rand((N,), generator=g) * 4.0 - 2.0).to(torch.float16 if dtype == 0 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("ks", [1, 2, 4])
@pytest.mark.parametrize("M,N,K,G", [(100, 776, 1024, 64), (200, 520, 2048, 128), (16, 264, 1024, 32)])
def test_swap_parity(cuda_lib, M, N, K, G, ks, sym, dtype, with_bias):
    w = cuda_lib
    p = make_problem(M, N, K, G, sym, dtype, seed=16000 + M + N + K + ks)
    d = to_device(p, w)
    b = seeded_bias(N, dtype, seed=N + ks) if with_bias else None
    bias = None if b is None else bits_to_tensor(b, dtype)
    out = forced(w, [128, 4, 3, 2, ks, 1],
                 lambda: w.w4a16_gemm_fused(d["x"], d["qweight"], d["scales"], d["qzeros"], G, bias=bias,
                                            path=PREFILL))
    y = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
    check_tolerance(out_values(out), oracle.epilogue(y, N, dtype, bias=b),
                    f"swapped M={M} N={N} K={K} G={G} KS={ks}")
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("ks", [1, 3, 8])
def test_swap_integer_exact(cuda_lib, ks):
    w = cuda_lib
    M, N, K, G = 160, 1000, 2048, 64
    p = make_problem(M, N, K, G, False, 1, seed=16100 + ks, x_kind="int4")
    p.scales[:] = 0x3F80                               # bf16 1.0: every partial sum is an exact integer
    d = to_device(p, w)
    run = lambda: w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G)
    plain = forced(w, [128, 4, 3, 2, ks, 0], run)
    swapped = forced(w, [128, 4, 3, 2, ks, 1], run)
    assert np.array_equal(tensor_to_bits(swapped), tensor_to_bits(plain))
    want = oracle.round_array(oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1), 1)
    assert np.array_equal(tensor_to_bits(swapped), want)
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("ks", [1, 2])
def test_swap_dense_integer_exact(cuda_lib, ks):
    w = cuda_lib
    M, N, K, G = 90, 520, 1024, 128
    p = make_problem(M, N, K, G, True, 1, seed=16200 + ks, x_kind="int4")
    p.scales[:] = 0x3F80
    d = to_device(p, w)
    cache = w.w4a16_dequantize(d["qweight"], d["scales"], d["qzeros"], G)
    plain = forced(w, [128, 4, 4, 2, ks, 0], lambda: w.w4a16_gemm_dense(d["x"], cache))
    swapped = forced(w, [128, 4, 4, 2, ks, 1], lambda: w.w4a16_gemm_dense(d["x"], cache))
    assert np.array_equal(tensor_to_bits(swapped), tensor_to_bits(plain))
    want = oracle.round_array(oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1), 1)
    assert np.array_equal(tensor_to_bits(swapped), want)
    assert w.w4a16_last_device_error() == 0
