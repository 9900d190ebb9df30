"""GPU parity of the fused epilogues (w4a16_gemm_fused) against the oracle:
the optional bias on both kernels and SiLU-and-multiply over a merged
gate/up weight on the decode kernel.

* bias: within the contract's tolerance on seeded inputs, and bit-exact on
  integer-exact inputs (s = 1, integer x and bias) for every decode
  configuration family and for the prefill kernel with and without a K split;
* SiLU-and-multiply: within tolerance, with and without bias, ragged I and
  K tails, clusters of 1 to 8 CTAs, both TMA forms (K a multiple of 128 or
  not), fp16 and bf16, symmetric and asymmetric, and on the full-size
  Qwen3-4B and Llama-3.1-8B gate_up layers.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import bits_to_tensor, check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

DECODE, PREFILL = 1, 2
EPI_NONE, EPI_SILU = 0, 1


def seeded_bias(N, dtype, seed, lo=-2.0, hi=2.0, integer=False):
    g = torch.Generator().manual_seed(seed)
    if integer:
        v = torch.randint(-8, 9, (N,), generator=g).to(torch.float32)
    else:
        v = torch.rand((N,), generator=g) * (hi - lo) + lo
    t = v.to(torch.float16 if dtype == 0 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def reference(p, d, bias_bits, silu):
    y = oracle.gemm(p.x, p.M, p.K, d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, p.dtype)
    return oracle.epilogue(y, p.N, p.dtype, bias=bias_bits, silu_mul=silu)


def run_fused(w, p, d, bias_bits, epi, path=0):
    bias = None if bias_bits is None else bits_to_tensor(bias_bits, p.dtype)
    out = w.w4a16_gemm_fused(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G, bias=bias,
                             epilogue=epi, path=path)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("M,N,K,G", [(1, 264, 1152, 128), (3, 1000, 1184, 32), (8, 520, 4096, 64),
                                     (5, 2048, 2560, 128)])
def test_decode_bias(cuda_lib, M, N, K, G, sym, dtype):
    w = cuda_lib
    p = make_problem(M, N, K, G, sym, dtype, seed=9100 + M + N + K)
    d = to_device(p, w)
    b = seeded_bias(N, dtype, seed=N + K)
    out = run_fused(w, p, d, b, EPI_NONE, path=DECODE)
    check_tolerance(out_values(out), reference(p, d, b, False), f"decode bias M={M} N={N} K={K}")


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("M,I,K,G", [(1, 132, 1152, 128), (2, 500, 1184, 32), (8, 260, 4096, 64),
                                     (4, 1024, 2560, 128)])
def test_decode_silu_mul(cuda_lib, M, I, K, G, with_bias, sym, dtype):
    w = cuda_lib
    N = 2 * I
    p = make_problem(M, N, K, G, sym, dtype, seed=9200 + M + I + K)
    d = to_device(p, w)
    b = seeded_bias(N, dtype, seed=I + K) if with_bias else None
    out = run_fused(w, p, d, b, EPI_SILU)
    assert tuple(out.shape) == (M, I)
    check_tolerance(out_values(out), reference(p, d, b, True), f"silu_mul M={M} I={I} K={K}")


DECODE_FORCED = [[1, 4, 4, 2, 5], [1, 8, 2, 3, 2], [2, 4, 2, 2, 3], [1, 4, 4, 4, 8], [1, 2, 4, 3, 7],
                 [2, 8, 1, 2, 2], [1, 4, 4, 2, 1]]


@pytest.mark.parametrize("cfg", DECODE_FORCED, ids=lambda c: "-".join(map(str, c)))
def test_decode_forced_configs(cuda_lib, cfg):
    """Every decode configuration family: bias bit-exact on integer-exact
    inputs; SiLU-and-multiply (with bias) within tolerance."""
    w = cuda_lib
    for (M, N, K, G, sym) in [(1, 264, 2560, 128, True), (3, 1000, 1184, 32, False), (8, 520, 4096, 64, False)]:
        p = make_problem(M, N, K, G, sym, 1, seed=9300 + M + N, x_kind="int4")
        p.scales[:] = 0x3F80
        d = to_device(p, w)
        b = seeded_bias(N, 1, seed=N, integer=True)
        w.w4a16_debug_set_config(1, cfg)
        try:
            out = run_fused(w, p, d, b, EPI_NONE, path=DECODE)
            want = oracle.round_array(reference(p, d, b, False), 1)
            assert np.array_equal(tensor_to_bits(out), want), (cfg, M, N, K)
            q = make_problem(M, N, K, G, sym, 1, seed=9400 + M + N)
            dq = to_device(q, w)
            bq = seeded_bias(N, 1, seed=N + 1)
            out = run_fused(w, q, dq, bq, EPI_SILU)
            check_tolerance(out_values(out), reference(q, dq, bq, True), f"silu {cfg} M={M} N={N} K={K}")
        finally:
            w.w4a16_debug_set_config(1, None)
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("M,N,K,G,ks", [(16, 520, 1152, 64, None), (200, 264, 2048, 128, None),
                                        (40, 1000, 4096, 32, 4), (130, 512, 2560, 128, 2)])
def test_prefill_bias(cuda_lib, M, N, K, G, ks, dtype):
    """Bias on the prefill kernel (TMA-store epilogue, and the K-split
    cluster reduction): tolerance on seeded inputs, bit-exact on
    integer-exact ones."""
    w = cuda_lib
    if ks is not None:
        w.w4a16_debug_set_config(2, [128, 3, 2, 2, ks])
    try:
        p = make_problem(M, N, K, G, False, dtype, seed=9500 + M + N)
        d = to_device(p, w)
        b = seeded_bias(N, dtype, seed=M + N)
        out = run_fused(w, p, d, b, EPI_NONE, path=PREFILL)
        check_tolerance(out_values(out), reference(p, d, b, False), f"prefill bias M={M} N={N} K={K} ks={ks}")
        q = make_problem(M, N, K, G, True, dtype, seed=9600 + M + N, x_kind="int4")
        q.scales[:] = 0x3C00 if dtype == 0 else 0x3F80
        dq = to_device(q, w)
        bq = seeded_bias(N, dtype, seed=M, integer=True)
        out = run_fused(w, q, dq, bq, EPI_NONE, path=PREFILL)
        assert np.array_equal(tensor_to_bits(out), oracle.round_array(reference(q, dq, bq, False), dtype))
    finally:
        w.w4a16_debug_set_config(2, None)
    assert w.w4a16_last_device_error() == 0


def test_fused_matches_plain_without_epilogue(cuda_lib):
    """No bias, no activation: the fused entry point is w4a16_gemm bit for bit."""
    w = cuda_lib
    for M in (1, 5, 64):
        p = make_problem(M, 1024, 2048, 128, False, 1, seed=9700 + M)
        d = to_device(p, w)
        a = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G)
        b = run_fused(w, p, d, None, EPI_NONE)
        assert torch.equal(a, b)


@pytest.mark.parametrize("name,N,K,G,sym,dtype", [("qwen3-4b gate_up", 19456, 2560, 128, True, 1),
                                                  ("llama-3.1-8b gate_up", 28672, 4096, 128, False, 0)])
def test_fullsize_gate_up_silu(cuda_lib, name, N, K, G, sym, dtype):
    """The full-size merged gate/up layers at M = 1 and 4 with the fused
    SiLU-and-multiply, every output against the oracle."""
    w = cuda_lib
    for M in (1, 4):
        p = make_problem(M, N, K, G, sym, dtype, seed=9800 + M)
        d = to_device(p, w)
        out = run_fused(w, p, d, None, EPI_SILU)
        check_tolerance(out_values(out), reference(p, d, None, True), f"{name} M={M}")
    assert w.w4a16_last_device_error() == 0
