"""GPU parity over the whole dispatch/crossover sweep: every M in
{1, 2, 3, 4, 5, 6, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096} x G in
{32, 64, 128} x {symmetric, asymmetric} x {fp16, bf16} on the full-size
N x K in {2560 x 9728, 19456 x 2560, 4096 x 14336} (576 cells), through the
dispatcher's own choice of kernel.  The oracle computes every column of a
sample of rows: the first, the last and 30 seeded random ones (all rows
when M <= 32).

The weights of one (shape, G, form, dtype) group are drawn once, with the
seed of the group's first cell; each M takes the first M rows of one seeded
[4096, K] activation matrix, so every cell still has its own M and shares
nothing else with the others but the weights."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import bits_to_tensor, check_tolerance, out_values, to_device
from w4a16_group_quantised_gb300.workloads import SWEEP_M, SWEEP_SHAPES, make_problem, sweep_cells

pytestmark = pytest.mark.gpu

GROUPS = [(si, G, sym, dtype) for si in range(len(SWEEP_SHAPES)) for G in (32, 64, 128)
          for sym in (True, False) for dtype in (0, 1)]


def first_seed(N, K, G, sym, dtype):
    for c in sweep_cells():
        if (c["N"], c["K"], c["G"], c["sym"], c["dtype"]) == (N, K, G, sym, dtype):
            return c["seed"]
    raise KeyError


@pytest.mark.parametrize("si,G,sym,dtype", GROUPS,
                         ids=[f"{SWEEP_SHAPES[s][0]}x{SWEEP_SHAPES[s][1]}-G{g}-{'sym' if y else 'asym'}-"
                              f"{'fp16' if t == 0 else 'bf16'}" for s, g, y, t in GROUPS])
def test_sweep_cells(cuda_lib, si, G, sym, dtype):
    w = cuda_lib
    N, K = SWEEP_SHAPES[si]
    Mmax = max(SWEEP_M)
    p = make_problem(Mmax, N, K, G, sym, dtype, seed=first_seed(N, K, G, sym, dtype))
    d = to_device(p, w)
    for M in SWEEP_M:
        x = d["x"][:M]
        out = w.w4a16_gemm(x, d["qweight"], d["scales"], d["qzeros"], G)
        torch.cuda.synchronize()
        if M <= 32:
            rows = np.arange(M, dtype=np.int32)
        else:
            rng = np.random.default_rng(1000 * si + M + G)
            rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 30)])).astype(np.int32)
        y_ref = oracle.gemm(p.x[:M], M, K, d["ref_qw"], p.scales, d["ref_qz"], G, N, dtype, rows=rows)
        check_tolerance(out_values(out)[rows], y_ref, f"N={N} K={K} G={G} sym={sym} dt={dtype} M={M}")
    assert w.w4a16_last_device_error() == 0
