"""GPU parity of the MoE grouped skinny GEMM (w4a16_moe_gemm) against the
oracle's moe_gemm: routed tokens with repeated experts, optional routing
weights, ragged N and K, every group size, both forms and dtypes, forced
decode configurations (bit-exact on integer-exact inputs), an out-of-range
expert id (status word, zero row, context still usable), routing read at run
time under graph replay, and Qwen3-30B-A3B-like expert shapes."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import bits_to_tensor, check_tolerance, out_values, tensor_to_bits
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu


def experts(w, E, N, K, G, sym, dtype, seed, x_kind="normal", unit_scale=False):
    ps = [make_problem(1, N, K, G, sym, dtype, seed=seed + e, x_kind=x_kind) for e in range(E)]
    if unit_scale:
        for p in ps:
            p.scales[:] = 0x3C00 if dtype == 0 else 0x3F80
    qw = np.stack([oracle.pack(p.q) for p in ps])
    sc = np.stack([p.scales for p in ps])
    qz = None if sym else np.stack([oracle.pack_zeros(p.z) for p in ps])
    dev = dict(qweight=torch.from_numpy(qw).cuda(), scales=bits_to_tensor(sc, dtype),
               qzeros=None if qz is None else torch.from_numpy(qz).cuda())
    # the library's own packing of the stack agrees with the oracle's
    q_all = torch.from_numpy(np.concatenate([p.q for p in ps])).cuda()
    assert np.array_equal(w.w4a16_pack(q_all).cpu().numpy().reshape(qw.shape), qw)
    return qw, sc, qz, dev


def routing(T, topk, E, seed, weights):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, topk)).astype(np.int32)
    if T * topk > 1:
        ids.flat[-1] = ids.flat[0]              # at least one repeated expert
    rw = rng.uniform(-1.5, 1.5, size=(T, topk)).astype(np.float32) if weights else None
    return ids, rw


def tokens(T, K, dtype, seed, x_kind="normal"):
    return make_problem(T, 8, K, 32, True, dtype, seed=seed, x_kind=x_kind).x


def run(w, xb, dtype, dev, G, ids, rw):
    x = bits_to_tensor(xb, dtype)
    out = w.w4a16_moe_gemm(x, dev["qweight"], dev["scales"], dev["qzeros"], G, torch.from_numpy(ids).cuda(),
                           route_weights=None if rw is None else torch.from_numpy(rw).cuda())
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("T,topk,E,N,K,G,weights", [(1, 1, 4, 264, 1184, 32, False), (3, 2, 8, 520, 2048, 64, True),
                                                   (8, 4, 6, 1000, 1152, 128, True), (5, 8, 16, 256, 4096, 128, False)])
def test_moe_parity(cuda_lib, T, topk, E, N, K, G, weights, sym, dtype):
    w = cuda_lib
    qw, sc, qz, dev = experts(w, E, N, K, G, sym, dtype, seed=15000 + E + N)
    ids, rw = routing(T, topk, E, seed=T * 7 + topk, weights=weights)
    xb = tokens(T, K, dtype, seed=15100 + T)
    out = run(w, xb, dtype, dev, G, ids, rw)
    assert tuple(out.shape) == (T, topk, N)
    ref = oracle.moe_gemm(xb, T, K, qw, sc, qz, G, N, ids, dtype, route_weights=rw)
    check_tolerance(out_values(out).reshape(T * topk, N), ref.reshape(T * topk, N),
                    f"moe T={T} topk={topk} E={E} N={N} K={K} G={G}")
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("cfg", [None, [1, 4, 4, 2, 1], [1, 8, 2, 3, 2], [2, 4, 2, 2, 3], [1, 2, 4, 3, 7]],
                         ids=lambda c: "auto" if c is None else "-".join(map(str, c)))
def test_moe_integer_exact(cuda_lib, cfg):
    w = cuda_lib
    T, topk, E, N, K, G = 4, 3, 5, 520, 2560, 128
    qw, sc, qz, dev = experts(w, E, N, K, G, False, 1, seed=15200, x_kind="int4", unit_scale=True)
    ids, _ = routing(T, topk, E, seed=3, weights=False)
    xb = tokens(T, K, 1, seed=15300, x_kind="int4")
    if cfg is not None:
        w.w4a16_debug_set_config(1, cfg)
    try:
        out = run(w, xb, 1, dev, G, ids, None)
    finally:
        w.w4a16_debug_set_config(1, None)
    want = oracle.round_array(oracle.moe_gemm(xb, T, K, qw, sc, qz, G, N, ids, 1), 1)
    assert np.array_equal(tensor_to_bits(out), want)
    assert w.w4a16_last_device_error() == 0


def test_moe_bad_expert_id(cuda_lib):
    """An id outside [0, E): that row is zero, the status word reads
    W4A16_ERR_ARG, the other rows are right, and the next call is clean."""
    w = cuda_lib
    T, topk, E, N, K, G = 2, 2, 3, 256, 1024, 128
    qw, sc, qz, dev = experts(w, E, N, K, G, True, 1, seed=15400)
    ids = np.array([[0, 7], [2, 1]], dtype=np.int32)
    xb = tokens(T, K, 1, seed=15500)
    w.w4a16_clear_device_error()
    out = run(w, xb, 1, dev, G, ids, None)
    assert w.w4a16_last_device_error() == -9
    w.w4a16_clear_device_error()
    vals = out_values(out)
    assert np.all(vals[0, 1] == 0.0)
    good = ids.copy()
    good[0, 1] = 0
    ref = oracle.moe_gemm(xb, T, K, qw, sc, qz, G, N, good, 1)
    for (t, j) in [(0, 0), (1, 0), (1, 1)]:
        check_tolerance(vals[t, j], ref[t, j], f"slot {t},{j}")
    out = run(w, xb, 1, dev, G, good, None)
    check_tolerance(out_values(out).reshape(-1, N), ref.reshape(-1, N), "after a bad id")
    assert w.w4a16_last_device_error() == 0


def test_moe_routing_read_at_run_time(cuda_lib):
    """Captured once, replayed with new expert ids written into the same
    device buffer: each replay follows the routing of that moment."""
    w = cuda_lib
    T, topk, E, N, K, G = 2, 4, 8, 512, 2048, 64
    qw, sc, qz, dev = experts(w, E, N, K, G, False, 1, seed=15600)
    xb = tokens(T, K, 1, seed=15700)
    x = bits_to_tensor(xb, 1)
    ids_dev = torch.zeros((T, topk), dtype=torch.int32, device="cuda")
    out = torch.empty((T, topk, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        w.w4a16_moe_gemm(x, dev["qweight"], dev["scales"], dev["qzeros"], G, ids_dev, out=out)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            w.w4a16_moe_gemm(x, dev["qweight"], dev["scales"], dev["qzeros"], G, ids_dev, out=out)
    for r in range(3):
        ids, _ = routing(T, topk, E, seed=100 + r, weights=False)
        with torch.cuda.stream(stream):
            ids_dev.copy_(torch.from_numpy(ids))
            g.replay()
        torch.cuda.synchronize()
        ref = oracle.moe_gemm(xb, T, K, qw, sc, qz, G, N, ids, 1)
        check_tolerance(out_values(out).reshape(-1, N), ref.reshape(-1, N), f"replay {r}")
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("name,N,K", [("experts gate_up", 1536, 2048), ("experts down", 2048, 768)])
def test_moe_expert_shapes(cuda_lib, name, N, K):
    """Qwen3-30B-A3B-like experts (128 experts, top-8, bf16, symmetric,
    G = 128) at T = 1 and 4 tokens, every output checked."""
    w = cuda_lib
    E, topk, G = 128, 8, 128
    qw, sc, qz, dev = experts(w, E, N, K, G, True, 1, seed=15800)
    for T in (1, 4):
        ids, rw = routing(T, topk, E, seed=T, weights=True)
        xb = tokens(T, K, 1, seed=15900 + T)
        out = run(w, xb, 1, dev, G, ids, rw)
        ref = oracle.moe_gemm(xb, T, K, qw, sc, qz, G, N, ids, 1, route_weights=rw)
        check_tolerance(out_values(out).reshape(-1, N), ref.reshape(-1, N), f"{name} T={T}")
    assert w.w4a16_last_device_error() == 0
