"""Child process of test_gpu_trace.py (not a test module): runs two M = 1
decode layers on the trace build of the library (W4A16_LIBRARY=trace) and
saves to the .npz path given: the outputs with the timeline off and on, the
timeline buffer, and the buffer after a further launch with the timeline
turned off (which must leave it zero)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import w4a16_group_quantised_gb300 as w  # noqa: E402
from parity_helpers import tensor_to_bits, to_device  # noqa: E402
from w4a16_group_quantised_gb300.workloads import make_problem  # noqa: E402

# (N, K, seed) of the two traced layers; test_gpu_trace.py uses the same
SHAPES = ((4096, 2560, 17000), (2560, 4096, 17001))


def main(path):
    assert os.environ.get("W4A16_LIBRARY") == "trace"
    w.load_library()
    assert w.library_path().endswith("libw4a16_trace.so")
    probs = [make_problem(1, N, K, 128, True, 1, seed=s) for N, K, s in SHAPES]
    devs = [to_device(p, w) for p in probs]

    def run():
        return [w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], p.G) for d, p in zip(devs, probs)]

    off = run()
    buf = w.w4a16_debug_decode_trace([(N, K) for N, K, _ in SHAPES])
    try:
        on = run()
        torch.cuda.synchronize()
        trace = buf.cpu().numpy()
    finally:
        w.w4a16_debug_decode_trace(None)
    buf.zero_()
    run()
    torch.cuda.synchronize()
    after = buf.cpu().numpy()
    np.savez(path, off0=tensor_to_bits(off[0]), off1=tensor_to_bits(off[1]), on0=tensor_to_bits(on[0]),
             on1=tensor_to_bits(on[1]), trace=trace, after=after,
             status=np.array([w.w4a16_last_device_error()]))


if __name__ == "__main__":
    main(sys.argv[1])
