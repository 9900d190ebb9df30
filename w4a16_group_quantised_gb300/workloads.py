"""Seeded synthetic inputs for the W4A16 linear layer.

This module only draws random numbers; it holds none of the layer's arithmetic
(no packing, no dequantisation, no products).  Both the CUDA path and the CPU
oracle receive exactly these arrays and pack them themselves.

Draw order (fixed): x (fp32 normal -> activation dtype), q (uniform integers
0..15, [N, K]), scales (fp32 uniform [lo, hi] -> activation dtype, [N, K/G]),
z (uniform integers 0..15, [N, K/G]; drawn for symmetric cells too, then
unused).  16-bit tensors are returned as uint16 bit patterns.

The shapes are the linear layers of the models the pages benchmark
("[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP skinny
decode", benchmark tables): real checkpoints are not used; synthetic tensors
of the same shapes and of the stated value distributions stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

F16, BF16 = 0, 1
_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}
DTYPE_NAME = {F16: "fp16", BF16: "bf16"}

# N x K of the four linear layers of each model family.
QWEN3_4B_SHAPES = [("qkv", 6144, 2560), ("o_proj", 2560, 4096),
                   ("gate_up", 19456, 2560), ("down", 2560, 9728)]
LLAMA31_8B_SHAPES = [("qkv", 6144, 4096), ("o_proj", 4096, 4096),
                     ("gate_up", 28672, 4096), ("down", 4096, 14336)]
SWEEP_SHAPES = [(2560, 9728), (19456, 2560), (4096, 14336)]
SWEEP_M = [1, 2, 3, 4, 5, 6, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096]


@dataclass
class Problem:
    M: int
    N: int
    K: int
    G: int
    sym: bool
    dtype: int
    x: np.ndarray        # uint16 [M, K]
    q: np.ndarray        # uint8 [N, K], values 0..15
    scales: np.ndarray   # uint16 [N, K/G]
    z: np.ndarray | None  # uint8 [N, K/G] or None when symmetric
    seed: int

    @property
    def n_groups(self) -> int:
        return self.K // self.G


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def make_problem(M: int, N: int, K: int, G: int, sym: bool, dtype: int, seed: int,
                 scale_lo: float = 0.002, scale_hi: float = 0.02,
                 x_kind: str = "normal") -> Problem:
    """Draw one problem.  x_kind="normal" gives x ~ N(0,1); "int4" gives
    integers uniform in [-4, 4] (for integer-exact checks)."""
    g = torch.Generator().manual_seed(int(seed))
    td = _TORCH_DTYPE[dtype]
    if x_kind == "normal":
        x = torch.randn((M, K), generator=g, dtype=torch.float32).to(td)
    elif x_kind == "int4":
        x = torch.randint(-4, 5, (M, K), generator=g, dtype=torch.int32).to(td)
    else:
        raise ValueError(x_kind)
    q = torch.randint(0, 16, (N, K), generator=g, dtype=torch.uint8)
    s = (torch.rand((N, K // G), generator=g, dtype=torch.float32)
         * (scale_hi - scale_lo) + scale_lo).to(td)
    z = torch.randint(0, 16, (N, K // G), generator=g, dtype=torch.uint8)
    return Problem(M=M, N=N, K=K, G=G, sym=sym, dtype=dtype, x=_bits(x), q=q.numpy(),
                   scales=_bits(s), z=None if sym else z.numpy(), seed=int(seed))


def tiny_symmetric(M: int = 1) -> Problem:
    """M x K=256 x N=128, G=32, symmetric, fp16, scales U[0.005, 0.02], seed 0."""
    return make_problem(M, 128, 256, 32, True, F16, 0, scale_lo=0.005, scale_hi=0.02)


def qwen3_4b_decode(shape_idx: int, M: int, seed: int | None = None) -> Problem:
    name, N, K = QWEN3_4B_SHAPES[shape_idx]
    s = seed if seed is not None else shape_idx * 5 + (M - 1)
    return make_problem(M, N, K, 128, True, BF16, s)


def llama31_8b_decode(shape_idx: int, M: int, seed: int | None = None) -> Problem:
    name, N, K = LLAMA31_8B_SHAPES[shape_idx]
    s = seed if seed is not None else shape_idx * 5 + (M - 1)
    return make_problem(M, N, K, 128, False, F16, s)


def llama31_8b_prefill(shape_idx: int, M: int, seed: int | None = None) -> Problem:
    name, N, K = LLAMA31_8B_SHAPES[shape_idx]
    s = seed if seed is not None else shape_idx * 2 + (0 if M == 128 else 1)
    return make_problem(M, N, K, 64, False, BF16, s)


def sweep_cells():
    """Enumerate the crossover-sweep cells in order: shape, M, G, sym, dtype."""
    idx = 0
    for (N, K) in SWEEP_SHAPES:
        for M in SWEEP_M:
            for G in (32, 64, 128):
                for sym in (True, False):
                    for dtype in (F16, BF16):
                        yield dict(M=M, N=N, K=K, G=G, sym=sym, dtype=dtype, seed=idx)
                        idx += 1
