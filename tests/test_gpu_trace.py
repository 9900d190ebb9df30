"""The decode kernel's timeline hook (w4a16_debug_decode_trace).

* The default library has no stamps compiled in: it refuses a buffer
  (W4A16_ERR_ARG) and accepts turning the hook off.
* The trace build (libw4a16_trace.so, run in a child process with
  W4A16_LIBRARY=trace): every CTA of a traced layer writes its events in
  time order, only cluster rank 0 writes the gather event, untraced layer
  slots stay empty, turning the hook off stops the writes, and its outputs,
  traced or not, are bit-equal to the default library's.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

from parity_helpers import tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SHAPES = ((4096, 2560, 17000), (2560, 4096, 17001))      # as in decode_trace_child.py
W4A16_ERR_ARG = -9


def test_default_build_refuses_a_trace_buffer(cuda_lib):
    w = cuda_lib
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_debug_decode_trace([(4096, 2560)])
    assert e.value.code == W4A16_ERR_ARG
    w.w4a16_debug_decode_trace(None)


def test_decode_trace_events(cuda_lib, tmp_path):
    w = cuda_lib
    from w4a16_group_quantised_gb300 import build as libbuild
    libbuild.build(variant="trace")
    out = tmp_path / "trace.npz"
    env = dict(os.environ, W4A16_LIBRARY="trace")
    r = subprocess.run([sys.executable, os.path.join(HERE, "decode_trace_child.py"), str(out)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    z = np.load(out)
    assert int(z["status"][0]) == 0

    probs = [make_problem(1, N, K, 128, True, 1, seed=s) for N, K, s in SHAPES]
    for i, p in enumerate(probs):
        d = to_device(p, w)
        ref = tensor_to_bits(w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G))
        assert np.array_equal(z[f"off{i}"], ref)
        assert np.array_equal(z[f"on{i}"], ref)

    tr = z["trace"]
    for li in range(len(SHAPES)):
        ctas = tr[li][tr[li][:, 0] > 0]
        assert len(ctas) > 0
        for c in ctas:
            t = c[[0, 1, 2, 3, 4, 6]]
            assert np.all(np.diff(t) >= 0), c          # entry <= release <= x <= first stage <= loop end <= exit
            if c[7] == 0:
                assert c[4] <= c[5] <= c[6]            # rank 0 gathers, then stores
            else:
                assert c[5] == 0
    assert tr[len(SHAPES):].max() == 0                   # untraced pairs stay empty
    assert int(np.abs(z["after"]).max()) == 0            # off: a new launch does not write
