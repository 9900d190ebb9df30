"""GPU parity of the balanced (stream-K) decode kernel, an option enabled
through the configuration hook (which = 4), against the CPU oracle.  The
kernel keeps cross-CTA partial sums in a per-device workspace and resets its
per-row-block tickets itself, so repeated calls must stay exact."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

DECODE = 1
# N x K: one row block, ragged row and K tails, more row blocks than SMs
SHAPES = [(8, 32), (136, 288), (264, 1024), (1000, 2560), (5128, 1184)]


def _gemm_sk(w, d, G, ns=4):
    w.w4a16_debug_set_config(4, [1, ns])
    try:
        out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=DECODE)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(4, None)
    return out


@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
def test_decode_sk_parity(cuda_lib, M, dtype, sym):
    for i, (N, K) in enumerate(SHAPES):
        for G in (32, 64, 128):
            if K % G:
                continue
            p = make_problem(M, N, K, G, sym, dtype, seed=5000 + 10 * i + G + M)
            d = to_device(p, cuda_lib)
            out = _gemm_sk(cuda_lib, d, G)
            y_ref = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
            check_tolerance(out_values(out), y_ref, f"sk M={M} N={N} K={K} G={G} sym={sym} dt={dtype}")


@pytest.mark.parametrize("ns", [2, 4, 6])
def test_decode_sk_integer_exact_repeated(cuda_lib, ns):
    """s = 1, x integer: bit-exact, on three calls in a row (the tickets must
    be back at zero after every call)."""
    w = cuda_lib
    for (N, K, G) in [(264, 2560, 128), (5128, 1184, 32)]:
        p = make_problem(5, N, K, G, False, 1, seed=5100 + N, x_kind="int4")
        p.scales[:] = 0x3F80
        d = to_device(p, w)
        y_ref = oracle.gemm(p.x, 5, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1)
        want = oracle.round_array(y_ref, 1)
        for _ in range(3):
            out = _gemm_sk(w, d, G, ns)
            assert np.array_equal(tensor_to_bits(out), want), (N, K, G, ns)
    assert w.w4a16_last_device_error() == 0
