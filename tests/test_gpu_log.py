"""W4A16_LOG: the GEMM entry points print the kernel they launched."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, torch
sys.path.insert(0, %r)
import w4a16_group_quantised_gb300 as w
from w4a16_group_quantised_gb300.workloads import make_problem
w.load_library()
for M in (1, 1, 64):
    p = make_problem(M, 256, 512, 128, True, 1, seed=1)
    q = w.w4a16_pack(torch.from_numpy(p.q).cuda())
    x = torch.from_numpy(p.x.view('int16')).view(torch.bfloat16).cuda()
    s = torch.from_numpy(p.scales.view('int16')).view(torch.bfloat16).cuda()
    w.w4a16_gemm(x, q, s, None, 128)
    w.w4a16_gemm_fused(x[:1], q, s, None, 128, epilogue=w.EPI_SILU_MUL)
torch.cuda.synchronize()
"""


def run(mode):
    env = dict(os.environ, W4A16_LOG=str(mode))
    r = subprocess.run([sys.executable, "-c", SCRIPT % ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stderr.splitlines() if l.startswith("w4a16: ")]


def test_log_once_per_selection(cuda_lib):
    lines = run(1)
    dec = [l for l in lines if "path=decode kernel=decode_kernel" in l and "epilogue=none" in l]
    silu = [l for l in lines if "epilogue=silu_mul" in l]
    pre = [l for l in lines if "path=prefill kernel=prefill_kernel" in l]
    assert len(dec) == 1 and "M=1 N=256 K=512 G=128 bf16 sym" in dec[0] and " S=" in dec[0]
    assert len(silu) == 1
    assert len(pre) == 1 and "M=64" in pre[0] and " BN=" in pre[0]


def test_log_every_call(cuda_lib):
    lines = run(2)
    assert len([l for l in lines if "epilogue=none" in l and "path=decode" in l]) == 2
    assert len(run(0)) == 0


SPLIT_SCRIPT = r"""
import sys, torch
sys.path.insert(0, %r)
import w4a16_group_quantised_gb300 as w
w.load_library()
M, N, K, G = 1920, 6144, 4096, 64
x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
qw = torch.randint(-2**31, 2**31 - 1, (N, K // 8), dtype=torch.int32, device="cuda")
s = (torch.rand(N, K // G, device="cuda") * 0.01 + 0.001).to(torch.bfloat16)
qz = torch.randint(-2**31, 2**31 - 1, (N // 8, K // G), dtype=torch.int32, device="cuda")
w.w4a16_gemm(x, qw, s, qz, G)
torch.cuda.synchronize()
"""


def test_log_prefill_row_split(cuda_lib):
    """The Llama-3.1-8B qkv layer at M = 1920 (192 wide tiles on 152 SMs)
    runs as two launches over two blocks of weight rows, and the log says
    so; the full-size parity test of that layer therefore checks both."""
    env = dict(os.environ, W4A16_LOG="1")
    r = subprocess.run([sys.executable, "-c", SPLIT_SCRIPT % ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    pre = [l for l in r.stderr.splitlines() if "path=prefill" in l]
    assert len(pre) == 1 and "rows 0.." in pre[0], pre
