"""GPU parity of the stream-K decode kernel (csrc/decode_stream.cu) against the
oracle, through the C ABI.

The kernel is forced with w4a16_debug_set_config(6, [2, D]).  Shapes are chosen
so that every reduction path runs: row blocks that one warp covers (stored
directly), row blocks split between the warps of a CTA (summed in shared
memory), row blocks split between CTAs (global partial slots and tickets),
grids with fewer units than warps, and row counts that are not a multiple of
the 32-row unit (zero-filled rows past N)."""
import threading

import numpy as np
import pytest
import torch

import oracle
from parity_helpers import check_tolerance, out_values, tensor_to_bits, to_device
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

DECODE = 1

# (N, K): K a multiple of 256 (the kernel's unit)
SHAPES = [(8, 256), (136, 256), (264, 512), (1000, 1024), (2056, 2560), (4104, 768), (520, 9728)]


def stream_applicable(M, K, G, sym):
    """The stream-K kernel's host-side condition: K a multiple of 256 and its
    shared memory (at least two 4 KB weight slots per warp, three units of
    metadata per warp, x staged whole, the warps' partial slots) within the
    110 KB that lets two CTAs share an SM."""
    if K % 256 or not 1 <= M <= 8:
        return False
    ms = 32 * (512 // G) + (0 if sym else 4 * (1024 // G))
    xp = (K * 2 + 127) // 128 * 128 + 64
    for D in (4, 3, 2):
        off = 8 * D * 4096 + 8 * 3 * ms
        off = (off + 15) // 16 * 16 + M * xp
        off = (off + 15) // 16 * 16 + 8 * 2 * 32 * M * 4
        off = (off + 15) // 16 * 16 + 8 * D * 8 + 16 + 4 * 17
        if off + 128 <= 110 * 1024:
            return True
    return False


def forced(w, mode, d=0):
    w.w4a16_debug_set_config(6, [mode, d] if d else [mode])


def reference(p, d):
    return oracle.gemm(p.x, p.M, p.K, d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, p.dtype)


@pytest.mark.parametrize("M", [1, 2, 5, 8])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
def test_stream_tolerance(cuda_lib, M, dtype, sym):
    w = cuda_lib
    forced(w, 2)
    try:
        for i, (N, K) in enumerate(SHAPES):
            for G in (32, 64, 128):
                if not stream_applicable(M, K, G, sym):
                    continue
                p = make_problem(M, N, K, G, sym, dtype, seed=31000 + 10 * i + G + M)
                d = to_device(p, w)
                out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=DECODE)
                torch.cuda.synchronize()
                check_tolerance(out_values(out), reference(p, d),
                                f"stream M={M} N={N} K={K} G={G} sym={sym} dt={dtype}")
    finally:
        w.w4a16_debug_set_config(6, None)
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("D", [2, 3, 4])
@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("dtype", [0, 1])
def test_stream_integer_exact(cuda_lib, D, sym, dtype):
    """s = 1 and integer x: every partial sum is exact, so the output equals
    the oracle's bit for bit whatever the split; run twice in a row (the
    tickets must be back at zero after each call)."""
    w = cuda_lib
    one = 0x3C00 if dtype == 0 else 0x3F80
    cases = [(1, 264, 2560, 128), (3, 1000, 1024, 32), (8, 520, 1024, 64), (1, 8, 256, 32),
             (2, 19456, 512, 128), (1, 2560, 9728, 128)]
    forced(w, 2, D)
    try:
        for (M, N, K, G) in cases:
            p = make_problem(M, N, K, G, sym, dtype, seed=32000 + M + N + K, x_kind="int4")
            p.scales[:] = one
            d = to_device(p, w)
            want = oracle.round_array(reference(p, d), dtype)
            for _ in range(2):
                out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], G, path=DECODE)
                torch.cuda.synchronize()
                assert np.array_equal(tensor_to_bits(out), want), (D, M, N, K, G)
    finally:
        w.w4a16_debug_set_config(6, None)
    assert w.w4a16_last_device_error() == 0


def test_stream_matches_cluster_kernel_on_integers(cuda_lib):
    """The two decode kernels agree bit for bit on integer-exact inputs."""
    w = cuda_lib
    p = make_problem(4, 1032, 2048, 64, False, 1, seed=33001, x_kind="int4")
    p.scales[:] = 0x3F80
    d = to_device(p, w)
    outs = []
    for mode in (1, 2):
        forced(w, mode)
        try:
            outs.append(tensor_to_bits(w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], 64,
                                                    path=DECODE)))
        finally:
            w.w4a16_debug_set_config(6, None)
    assert np.array_equal(outs[0], outs[1])


def test_stream_repeatable_full_size(cuda_lib):
    """Qwen3-4B gate_up shape at M = 1 (bf16, G = 128): five calls in a row give
    identical bits (deterministic reduction order), within tolerance of the
    oracle."""
    w = cuda_lib
    p = make_problem(1, 19456, 2560, 128, True, 1, seed=33002)
    d = to_device(p, w)
    first = None
    for _ in range(5):
        out = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], None, 128, path=DECODE)
        bits = tensor_to_bits(out)
        if first is None:
            first = bits
        assert np.array_equal(bits, first)
    check_tolerance(out_values(out), reference(p, d), "gate_up")


def test_stream_two_streams(cuda_lib):
    """Calls on two streams at once use separate scratch: both results are
    right (each stream's first call makes its scratch)."""
    w = cuda_lib
    probs = [make_problem(2, 2056, 2560, 128, s, 1, seed=33003 + s) for s in (True, False)]
    devs = [to_device(p, w) for p in probs]
    refs = [reference(p, d) for p, d in zip(probs, devs)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [None, None]

    def run(i):
        with torch.cuda.stream(streams[i]):
            for _ in range(20):
                outs[i] = w.w4a16_gemm(devs[i]["x"], devs[i]["qweight"], devs[i]["scales"], devs[i]["qzeros"],
                                       128, path=DECODE, stream=streams[i])
    ts = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    torch.cuda.synchronize()
    for i in range(2):
        check_tolerance(out_values(outs[i]), refs[i], f"stream {i}")


def test_stream_capture_without_scratch_falls_back(cuda_lib):
    """A decode call first made on a stream while it is being captured must
    not allocate: it runs the cluster kernel instead, and the graph's result
    is right."""
    w = cuda_lib
    p = make_problem(1, 1032, 2560, 128, True, 1, seed=33004)
    d = to_device(p, w)
    s = torch.cuda.Stream()
    out = torch.empty((1, 1032), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            w.w4a16_gemm(d["x"], d["qweight"], d["scales"], None, 128, out=out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    check_tolerance(out_values(out), reference(p, d), "captured first call")
