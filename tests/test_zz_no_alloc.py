"""The allocation-free decode entry point (static device scratch), through
the C ABI, against the existing entry point on the same inputs: two calls
in a row must both equal w4a16_gemm with the same (balanced) decode kernel
bit for bit, and stay within the contract's tolerance of the oracle.  This
file is collected last so that it also runs after every other test."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M, N, K, G, sym, dtype", [
    (1, 6144, 2560, 128, True, 1),
    (5, 4096, 4096, 128, False, 0),
    (8, 5128, 1184, 32, False, 1),
])
def test_noalloc_matches_existing_entry_point(cuda_lib, M, N, K, G, sym, dtype):
    w = cuda_lib
    p = make_problem(M, N, K, G, sym, dtype, seed=6000 + M + N)
    d = to_device(p, w)
    td = torch.float16 if dtype == 0 else torch.bfloat16
    outs = [torch.empty((M, N), dtype=td, device="cuda") for _ in range(2)]
    for o in outs:                                   # two calls in a row
        w.w4a16_gemm_decode_noalloc(d["x"], d["qweight"], d["scales"], d["qzeros"], G, out=o)
    torch.cuda.synchronize()
    w.w4a16_debug_set_config(4, [1, 4])              # the same kernel through w4a16_gemm
    try:
        ref = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=1)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(4, None)
    for o in outs:
        assert np.array_equal(tensor_to_bits(o), tensor_to_bits(ref))
    y_ref = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
    check_tolerance(out_values(outs[1]), y_ref, f"noalloc M={M} N={N} K={K}")
    assert w.w4a16_last_device_error() == 0
