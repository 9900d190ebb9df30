"""The bounded-wait error path, made to run out on purpose without a fault:
with the test hook on, the decode kernel issues no weight copies, so every
CTA's wait for them ends at its time limit; the kernel leaves, the status word
reads W4A16_ERR_TIMEOUT, and the context stays usable -- the next call,
with the hook off, is correct again."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import check_tolerance, out_values, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

W4A16_ERR_TIMEOUT = -8


@pytest.mark.parametrize("cfg", [None, [1, 4, 4, 2, 1]], ids=["cluster", "single-cta"])
def test_bounded_wait_runs_out_and_context_survives(cuda_lib, cfg):
    w = cuda_lib
    p = make_problem(1, 256, 2560, 128, False, 1, seed=77)
    d = to_device(p, w)
    w.w4a16_clear_device_error()
    assert w.w4a16_last_device_error() == 0
    if cfg is not None:
        w.w4a16_debug_set_config(1, cfg)
    w.w4a16_debug_set_config(7, [1])
    try:
        w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G, path=1)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(7, None)
    assert w.w4a16_last_device_error() == W4A16_ERR_TIMEOUT
    w.w4a16_clear_device_error()
    assert w.w4a16_last_device_error() == 0
    try:
        out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G, path=1)
        torch.cuda.synchronize()
    finally:
        if cfg is not None:
            w.w4a16_debug_set_config(1, None)
    ref = oracle.gemm(p.x, p.M, p.K, d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, p.dtype)
    check_tolerance(out_values(out), ref, "after the timeout")
    assert w.w4a16_last_device_error() == 0
