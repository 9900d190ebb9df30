"""Shared helpers of the GPU parity tests: move a seeded Problem to the
device (packing it with the library's own pack kernels), run the CUDA path,
and compare with the oracle under the contract's tolerances."""
import numpy as np
import torch

import oracle

# Contract: |y - y_ref| <= ATOL_REL * max(1, |y_ref|) elementwise, and
# ||y - y_ref||_2 / ||y_ref||_2 <= REL_L2.
ATOL_REL = 1e-2
REL_L2 = 5e-3

TORCH_DT = {0: torch.float16, 1: torch.bfloat16}


def bits_to_tensor(bits: np.ndarray, dtype: int, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DT[dtype]).to(device)


def tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_device(p, lib):
    """Pack q and z on the GPU with the library and check the packed words
    against the oracle's packing (bit-exact)."""
    q = torch.from_numpy(p.q).cuda()
    qweight = lib.w4a16_pack(q)
    ref_qw = oracle.pack(p.q)
    assert np.array_equal(qweight.cpu().numpy(), ref_qw), "w4a16_pack differs from oracle"
    qzeros = None
    ref_qz = None
    if p.z is not None:
        z = torch.from_numpy(p.z).cuda()
        qzeros = lib.w4a16_pack_zeros(z)
        ref_qz = oracle.pack_zeros(p.z)
        assert np.array_equal(qzeros.cpu().numpy(), ref_qz), "w4a16_pack_zeros differs from oracle"
    x = bits_to_tensor(p.x, p.dtype)
    scales = bits_to_tensor(p.scales, p.dtype)
    return dict(x=x, qweight=qweight, scales=scales, qzeros=qzeros, ref_qw=ref_qw, ref_qz=ref_qz)


def out_values(out: torch.Tensor) -> np.ndarray:
    return out.detach().float().cpu().numpy().astype(np.float64)


def check_tolerance(y: np.ndarray, y_ref: np.ndarray, what: str = ""):
    err = np.abs(y - y_ref)
    bound = ATOL_REL * np.maximum(1.0, np.abs(y_ref))
    bad = err > bound
    assert not np.any(~np.isfinite(y)), f"{what}: non-finite outputs"
    assert not bad.any(), (
        f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; worst err "
        f"{err.max():.4g} at {np.unravel_index(err.argmax(), err.shape)}")
    denom = np.linalg.norm(y_ref)
    if denom > 0:
        rel = np.linalg.norm(y - y_ref) / denom
        assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3g} > {REL_L2}"
