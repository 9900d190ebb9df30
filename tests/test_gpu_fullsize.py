"""GPU parity at the benchmark's full sizes, in the launch configuration the
benchmark times (the dispatcher's own choice): the Qwen3-4B-shaped symmetric
bf16 decode layers, the Llama-3.1-8B-shaped asymmetric fp16 decode layers
(M = 1..5, every output checked), and the Llama-3.1-8B-shaped asymmetric
bf16 G=64 prefill layers at M = 128 and M = 1920 (sampled rows: the first,
the last and 14 seeded random ones, every column)."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import check_tolerance, out_values, to_device
from w4a16_group_quantised_gb300.workloads import (LLAMA31_8B_SHAPES, QWEN3_4B_SHAPES,
                                                   llama31_8b_decode, llama31_8b_prefill,
                                                   qwen3_4b_decode)

pytestmark = pytest.mark.gpu


def _check(w, p, rows=None):
    d = to_device(p, w)
    out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G)
    torch.cuda.synchronize()
    y = out_values(out)
    y_ref = oracle.gemm(p.x, p.M, p.K, d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, p.dtype,
                        rows=rows)
    if rows is not None:
        y = y[rows]
    check_tolerance(y, y_ref, f"M={p.M} N={p.N} K={p.K}")


@pytest.mark.parametrize("shape", range(4))
def test_qwen3_4b_decode(cuda_lib, shape):
    for M in (1, 2, 3, 4, 5):
        _check(cuda_lib, qwen3_4b_decode(shape, M))


@pytest.mark.parametrize("shape", range(4))
def test_llama31_8b_decode(cuda_lib, shape):
    for M in (1, 2, 3, 4, 5):
        _check(cuda_lib, llama31_8b_decode(shape, M))


@pytest.mark.parametrize("M", [128, 1920])
@pytest.mark.parametrize("shape", range(4))
def test_llama31_8b_prefill(cuda_lib, shape, M):
    p = llama31_8b_prefill(shape, M)
    rng = np.random.default_rng(shape * 10 + M)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 14)])).astype(np.int32)
    _check(cuda_lib, p, rows=rows)


@pytest.mark.parametrize("shape", [0, 2, 3])
def test_llama31_8b_prefill_repeatable(cuda_lib, shape):
    """Repeated launches on the same inputs give the same bits (the prefill
    kernel's reduction order is fixed, so any difference is a hazard).  The
    qkv shape runs as two launches over two blocks of weight rows."""
    w = cuda_lib
    p = llama31_8b_prefill(shape, 1920)
    d = to_device(p, w)
    first = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G)
    for _ in range(6):
        again = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G)
        torch.cuda.synchronize()
        diff = (again.view(torch.int16) != first.view(torch.int16))
        assert not bool(diff.any()), f"{int(diff.sum())} outputs differ between launches"
    assert w.w4a16_last_device_error() == 0
