"""Host logic of the prefill dispatcher, without a GPU: the launch plan
(tile width BN, ring depths, K split, swapped operands, row split) through
the w4a16_debug_prefill_plan test hook, for a 152-SM device whose prefill
kernel keeps CLUSTERS[k - 1] clusters of k CTAs resident (one CTA per SM;
clusters of 2, 4 and 8 cover 152, 144 and 120 SMs).

* the Llama-3.1-8B layers at M = 1920: qkv (192 tiles of 240 tokens on 152
  SMs) splits its weight rows after one full wave, gate_up does not;
* invariants over a grid of shapes, both forms: the row split, the tile
  and ring parameters within the kernel's limits and its shared memory,
  room for the K-split partial tile, swapped operands only for 128-token
  tiles of the fused form.
"""
import ctypes
import itertools

import pytest

CLUSTERS = [152, 76, 48, 36, 24, 24, 16, 15]
SMEM_CAP = 227 * 1024


@pytest.fixture(scope="module")
def lib():
    from w4a16_group_quantised_gb300 import build
    build.build()
    import w4a16_group_quantised_gb300 as w
    return w.load_library()


def plan(lib, M, N, K, dense=False, clusters=CLUSTERS):
    out = (ctypes.c_int * 13)()
    cl = (ctypes.c_int * 8)(*clusters)
    rc = lib.w4a16_debug_prefill_plan(M, N, K, 1 if dense else 0, 152, cl, out)
    assert rc == 0, rc
    v = list(out)
    cfg = lambda o: dict(BN=v[o], SX=v[o + 1], SA=v[o + 2], SW=v[o + 3], KS=v[o + 4], swap=v[o + 5])
    return v[0], cfg(1), cfg(7)


def rings_bytes(c):
    # x ring (BN x 128 B a stage), rounded up to 1 KB; A ring (256 rows x 128 B); packed ring (256 x 128 B)
    x = (c["SX"] * c["BN"] * 128 + 1023) // 1024 * 1024
    return x + c["SA"] * 32768 + c["SW"] * 32768


def check_cfg(c, dense):
    assert 16 <= c["BN"] <= 256 and c["BN"] % 16 == 0
    assert 2 <= c["SX"] <= 6 and 2 <= c["SA"] <= 4
    assert 1 <= c["KS"] <= 8
    assert c["SW"] == (0 if dense else 2)
    rings = rings_bytes(c)
    bars = (2 * (c["SX"] + c["SA"] + c["SW"]) + 1) * 8 + 16
    assert rings + bars + 1024 <= SMEM_CAP, c
    # the epilogue stages a [BN][256] output tile over the x and A rings
    assert c["BN"] * 256 * 2 <= c["SX"] * c["BN"] * 128 + c["SA"] * 32768, c
    if c["KS"] > 1:                                  # fp32 partial tile over the rings
        assert c["BN"] * 256 * 4 <= rings, c
    assert c["swap"] in (0, 1)
    if c["swap"]:
        assert c["BN"] == 128 and not dense and c["KS"] <= 3, c


def test_llama_prefill_plans(lib):
    n_split, main, tail = plan(lib, 1920, 6144, 4096)          # qkv
    assert n_split == 4864                                       # 19 n-tiles x 8 m-tiles = one full wave
    assert main["BN"] == 240 and main["KS"] == 1 and main["swap"] == 0
    check_cfg(main, False)
    check_cfg(tail, False)
    n_split, main, _ = plan(lib, 1920, 28672, 4096)             # gate_up: whole waves already
    assert n_split == 28672 and main["BN"] == 240 and main["KS"] == 1
    n_split, main, _ = plan(lib, 1920, 4096, 14336)             # down: x of 55 MB keeps a 3-deep x ring
    assert n_split == 4096 and main["SX"] >= 3


@pytest.mark.parametrize("dense", [False, True])
def test_plan_invariants(lib, dense):
    for M, N, K in itertools.product((1, 16, 100, 128, 256, 640, 1920, 4096),
                                     (256, 520, 4096, 6144, 28672), (512, 4096, 14336)):
        n_split, main, tail = plan(lib, M, N, K, dense)
        assert 0 < n_split <= N
        check_cfg(main, dense)
        if n_split < N:
            assert n_split % 256 == 0
            assert main["KS"] == 1                               # whole waves of unsplit tiles
            check_cfg(tail, dense)


def test_plan_hook_rejects_bad_arguments(lib):
    out = (ctypes.c_int * 13)()
    cl = (ctypes.c_int * 8)(*CLUSTERS)
    assert lib.w4a16_debug_prefill_plan(0, 256, 512, 0, 152, cl, out) == -9
    assert lib.w4a16_debug_prefill_plan(16, 260, 512, 0, 152, cl, out) == -9   # N % 8
    assert lib.w4a16_debug_prefill_plan(16, 256, 512, 0, 0, cl, out) == -9     # no SMs
    bad = (ctypes.c_int * 8)(*([152, -1] + CLUSTERS[2:]))
    assert lib.w4a16_debug_prefill_plan(16, 256, 512, 0, 152, bad, out) == -9
    assert lib.w4a16_debug_prefill_plan(16, 256, 512, 0, 152, None, out) == -9
