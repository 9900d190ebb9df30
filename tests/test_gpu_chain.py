"""GPU tests of chained layers (w4a16_gemm_chain): layer i's output is layer
i+1's input, launched back to back with programmatic dependent launch, eagerly
and captured in a CUDA graph.  Every layer is checked against the oracle run on
the GPU's own output bits of the previous layer (so each comparison sees the
same input), which also checks the kernels' ordering: weights may be read
early, the input only after the previous kernel completed.

Also: weights packed on a stream and used by the very next GEMM on that
stream, without a synchronisation in between.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import (bits_to_tensor, check_tolerance, out_values, tensor_to_bits, to_device)
from w4a16_group_quantised_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu

EPI_NONE, EPI_SILU = 0, 1


def chain_layers(w, M, dtype, seed, silu=True):
    """A four-layer chain shaped like a transformer block's projections,
    scaled down: 1024 -> 1536 -> 1024 -> [gate | up] 2 x 1408 (SiLU-and-
    multiply: 1408) -> 1024, asymmetric and symmetric layers, G = 128 / 64."""
    gate_n = 2 * 1408
    down_k = 1408 if silu else gate_n
    specs = [(1536, 1024, 128, True, EPI_NONE, True), (1024, 1536, 64, False, EPI_NONE, False),
             (gate_n, 1024, 128, False, EPI_SILU if silu else EPI_NONE, True),
             (1024, down_k, 128, True, EPI_NONE, True)]
    layers = []
    for i, (N, K, G, sym, epi, with_bias) in enumerate(specs):
        p = make_problem(1, N, K, G, sym, dtype, seed=seed + i)
        d = to_device(p, w)
        bias_bits = None
        if with_bias:
            g = torch.Generator().manual_seed(seed + 100 + i)
            bt = (torch.rand((N,), generator=g) * 0.5 - 0.25).to(torch.float16 if dtype == 0 else torch.bfloat16)
            bias_bits = bt.view(torch.int16).numpy().view(np.uint16)
        layers.append(dict(p=p, d=d, qweight=d["qweight"], scales=d["scales"], qzeros=d["qzeros"], G=G,
                           epilogue=epi, bias_bits=bias_bits,
                           bias=None if bias_bits is None else bits_to_tensor(bias_bits, dtype)))
    return layers


def input_x(M, K, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((M, K), generator=g).to(torch.float16 if dtype == 0 else torch.bfloat16).cuda()


def check_layer_by_layer(x, layers, outs, dtype, what):
    inp = tensor_to_bits(x)
    for i, (L, out) in enumerate(zip(layers, outs)):
        p, d = L["p"], L["d"]
        M, K = inp.shape
        y = oracle.gemm(inp, M, K, d["ref_qw"], p.scales, d["ref_qz"], p.G, p.N, dtype)
        ref = oracle.epilogue(y, p.N, dtype, bias=L["bias_bits"], silu_mul=L["epilogue"] == EPI_SILU)
        check_tolerance(out_values(out), ref, f"{what} layer {i}")
        inp = tensor_to_bits(out)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("M", [1, 3, 8, 24, 200])
def test_chain_layer_by_layer(cuda_lib, M, dtype):
    w = cuda_lib
    layers = chain_layers(w, M, dtype, seed=11000 + M, silu=M <= 8)
    x = input_x(M, 1024, dtype, seed=M)
    outs = w.w4a16_gemm_chain(x, layers)
    torch.cuda.synchronize()
    check_layer_by_layer(x, layers, outs, dtype, f"chain M={M}")
    assert w.w4a16_last_device_error() == 0


@pytest.mark.parametrize("M", [1, 4])
def test_chain_in_cuda_graph(cuda_lib, M):
    """The chain captured once and replayed with new inputs copied into the
    captured input buffer: every replay equals the eager chain on the same
    input bit for bit, and the first one is checked layer by layer."""
    w = cuda_lib
    dtype = 1
    layers = chain_layers(w, M, dtype, seed=12000 + M)
    for L in layers:
        N = L["qweight"].shape[0]
        cols = N // 2 if L["epilogue"] == EPI_SILU else N
        L["out"] = torch.empty((M, cols), dtype=torch.bfloat16, device="cuda")
    x_static = torch.empty((M, 1024), dtype=torch.bfloat16, device="cuda")
    x_static.copy_(input_x(M, 1024, dtype, seed=0))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        w.w4a16_gemm_chain(x_static, layers)          # first calls outside capture (device set-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            w.w4a16_gemm_chain(x_static, layers)
    for r in range(3):
        xr = input_x(M, 1024, dtype, seed=100 + r)
        with torch.cuda.stream(stream):
            x_static.copy_(xr)
            g.replay()
        torch.cuda.synchronize()
        replayed = [L["out"].clone() for L in layers]
        if r == 0:
            check_layer_by_layer(xr, layers, replayed, dtype, f"graph replay M={M}")
        fresh = [dict(L, out=None) for L in layers]
        eager = w.w4a16_gemm_chain(xr, fresh)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(replayed, eager)):
            assert torch.equal(a, b), f"replay {r} layer {i} differs from the eager chain"
    assert w.w4a16_last_device_error() == 0


def test_pack_then_gemm_same_stream(cuda_lib):
    """New weights packed into the same buffer and used by the next GEMM on
    the same stream, with no synchronisation between them, three times over:
    each GEMM sees the weights just packed."""
    w = cuda_lib
    N, K, G = 1024, 2048, 128
    qweight = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
    qzeros = torch.empty((N // 8, K // G), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    for r in range(3):
        p = make_problem(2, N, K, G, False, 1, seed=13000 + r)
        q = torch.from_numpy(p.q).cuda()
        z = torch.from_numpy(p.z).cuda()
        x = bits_to_tensor(p.x, 1)
        s = bits_to_tensor(p.scales, 1)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            w.w4a16_pack(q, qweight=qweight, stream=stream)
            w.w4a16_pack_zeros(z, qzeros=qzeros, stream=stream)
            out = w.w4a16_gemm(x, qweight, s, qzeros, G, stream=stream)
        stream.synchronize()
        ref = oracle.gemm(p.x, 2, K, oracle.pack(p.q), p.scales, oracle.pack_zeros(p.z), G, N, 1)
        check_tolerance(out_values(out), ref, f"pack then gemm round {r}")
    assert w.w4a16_last_device_error() == 0
