"""GPU parity of the per-warp-stream decode kernel (K a multiple of 128; an
option enabled through the configuration hook) against the CPU oracle: the built-in configuration on shapes with ragged row
tails, and every forced configuration family (cell width, cluster split,
warps per CTA, ring depth), with the contract's tolerances and, on
integer-exact inputs, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.binding import W4A16Error
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

DECODE = 1
# N x K, K % 128 == 0; N covers one partial row unit, ragged unit tails, and
# more row units than SMs.
SHAPES = [(8, 128), (136, 384), (264, 1024), (1000, 2560), (5128, 1152)]


def _run(w, p, forced=None):
    w.w4a16_debug_set_config(5, [2] + list(forced) if forced is not None else [1])
    try:
        d = to_device(p, w)
        out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G, path=DECODE)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(5, None)
    return d, out


@pytest.mark.parametrize("M", [1, 2, 5, 8])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
def test_decode_warp_default(cuda_lib, M, dtype, sym):
    for i, (N, K) in enumerate(SHAPES):
        for G in (32, 64, 128):
            p = make_problem(M, N, K, G, sym, dtype, seed=3000 + 10 * i + G + M)
            d, out = _run(cuda_lib, p)
            y_ref = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype)
            check_tolerance(out_values(out), y_ref, f"M={M} N={N} K={K} G={G} sym={sym} dt={dtype}")


CONFIGS = [(nbk, s, nw, nsw) for nbk in (1, 2, 4) for s in (1, 2, 3, 8) for nw in (4, 8)
           for nsw in (1, 2, 3) if nsw * nbk >= 2]


@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_decode_warp_forced_configs(cuda_lib, M, sym):
    """Integer-exact inputs (s = 1, x in [-4, 4]): every configuration that
    the library accepts must give the rounded exact result bit for bit."""
    w = cuda_lib
    ran = 0
    for (N, K, G) in [(264, 2048, 64), (1000, 1024, 128)]:
        p = make_problem(M, N, K, G, sym, 1, seed=4100 + N + M, x_kind="int4")
        p.scales[:] = 0x3F80
        d = to_device(p, w)
        y_ref = oracle.gemm(p.x, M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, 1)
        want = oracle.round_array(y_ref, 1)
        for cfg in CONFIGS:
            w.w4a16_debug_set_config(5, [2] + list(cfg))
            try:
                out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=DECODE)
                torch.cuda.synchronize()
            except W4A16Error as e:
                assert e.code == -9, (cfg, e.code)   # configuration rejected for this shape
                continue
            finally:
                w.w4a16_debug_set_config(5, None)
            assert np.array_equal(tensor_to_bits(out), want), (N, K, G, cfg)
            ran += 1
    assert ran >= len(CONFIGS)


def test_decode_warp_matches_cluster_kernel(cuda_lib):
    """The two decode kernels agree within the contract on the same inputs
    (the cluster kernel is forced through its own configuration hook)."""
    w = cuda_lib
    p = make_problem(4, 2568, 3072, 128, False, 0, seed=4200)
    d, a = _run(w, p)
    w.w4a16_debug_set_config(1, [1, 4, 4, 4, 4])
    try:
        b = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 128, path=DECODE)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(1, None)
    check_tolerance(out_values(a), out_values(b).astype(np.float64), "warp vs cluster")


def test_decode_warp_deterministic(cuda_lib):
    w = cuda_lib
    p = make_problem(7, 4104, 2560, 32, False, 1, seed=4300)
    d, a = _run(w, p)
    w.w4a16_debug_set_config(5, [1])
    try:
        b = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 32, path=DECODE)
        torch.cuda.synchronize()
    finally:
        w.w4a16_debug_set_config(5, None)
    assert np.array_equal(tensor_to_bits(a), tensor_to_bits(b))
    assert w.w4a16_last_device_error() == 0
