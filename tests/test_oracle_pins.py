"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against something it does not compute itself:
hand-worked values (tests/golden), IEEE-754 decoding/rounding by numpy and
torch, an independent numpy restatement of unpacking, integer arithmetic that
is exact in any order, and a float64 library matmul.
"""
import numpy as np
import pytest
import torch

import oracle
from golden_cases import CASES, load, to_bits
from w4a16_group_quantised_gb300.workloads import make_problem

F16, BF16 = 0, 1


# --------------------------------------------------------------------- formats
def test_half_decode_all_patterns_fp16():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bits_to_float64(bits, F16)
    ref = bits.view(np.float16).astype(np.float64)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_half_decode_all_patterns_bf16():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bits_to_float64(bits, BF16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_round_trip_every_finite_pattern(dtype):
    bits = np.arange(65536, dtype=np.uint16)
    vals = oracle.bits_to_float64(bits, dtype)
    fin = np.isfinite(vals)
    back = oracle.round_array(vals[fin], dtype)
    assert np.array_equal(back, bits[fin])          # signed zeros included


def _bf16_rne_from_f32(v32: np.ndarray) -> np.ndarray:
    """Independent bf16 RN-even: add 0x7FFF plus the kept LSB, truncate."""
    u = v32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_exhaustive_product_rounding(dtype):
    """All 31 values of q - z times every finite 16-bit scale: the oracle's
    RN_dtype((q - z) * s) equals numpy's float16 cast (fp16) and both torch's
    bfloat16 cast and a bit-level RN-even (bf16).  Products have at most 15
    significant bits, so they are exact in float32 before the final rounding."""
    d = np.arange(-15, 16, dtype=np.int32)
    table = oracle.round_products(d, dtype)
    bits = np.arange(65536, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        if dtype == F16:
            s = bits.view(np.float16).astype(np.float64)
        else:
            s = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(s)
    for i, di in enumerate(d):
        prod = (float(di) * s[fin])
        if dtype == F16:
            with np.errstate(over="ignore"):
                ref = prod.astype(np.float16).view(np.uint16)
        else:
            with np.errstate(over="ignore"):
                p32 = prod.astype(np.float32)
            f32 = np.isfinite(p32)
            assert np.array_equal(p32[f32].astype(np.float64), prod[f32])  # exact in fp32
            ref = torch.from_numpy(p32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            ref2 = _bf16_rne_from_f32(p32)
            finite_ref = np.isfinite(p32)
            assert np.array_equal(ref[finite_ref], ref2[finite_ref])
        got = table[i][fin]
        # NaN payloads are not part of the contract; everything here is finite or inf
        assert np.array_equal(got, ref), f"d={di}"


def test_rounding_ties_go_to_even():
    # 1 + 2^-11 lies exactly between 1 and 1 + 2^-10 in fp16: ties to 1.0 (even)
    assert oracle.double_to_half(1.0 + 2.0 ** -11, F16) == 0x3C00
    # 1 + 3*2^-11 lies between 1+2^-10 (odd) and 1+2^-9 (even): goes up
    assert oracle.double_to_half(1.0 + 3 * 2.0 ** -11, F16) == 0x3C02
    # bf16: 1 + 2^-8 ties to 1.0, 1 + 3*2^-8 ties up to 1 + 2^-6
    assert oracle.double_to_half(1.0 + 2.0 ** -8, BF16) == 0x3F80
    assert oracle.double_to_half(1.0 + 3 * 2.0 ** -8, BF16) == 0x3F82
    # overflow and the largest finite value
    assert oracle.double_to_half(65504.0, F16) == 0x7BFF
    assert oracle.double_to_half(65520.0, F16) == 0x7C00
    # smallest fp16 subnormal and half of it (tie to zero)
    assert oracle.double_to_half(2.0 ** -24, F16) == 0x0001
    assert oracle.double_to_half(2.0 ** -25, F16) == 0x0000
    assert oracle.double_to_half(-0.0, F16) == 0x8000


# --------------------------------------------------------------------- packing
def test_pack_unpack_round_trip_random_q():
    rng = np.random.default_rng(1)
    q = rng.integers(0, 16, size=(24, 96), dtype=np.uint8)
    qw = oracle.pack(q)
    assert qw.shape == (24, 12) and qw.dtype == np.int32
    assert np.array_equal(oracle.unpack(qw, 96), q)
    assert np.array_equal(oracle.np_unpack(qw, 96), q)


def test_unpack_pack_round_trip_random_words():
    rng = np.random.default_rng(2)
    words = rng.integers(-2 ** 31, 2 ** 31, size=(16, 8), dtype=np.int64).astype(np.int32)
    q = oracle.unpack(words, 64)
    assert np.array_equal(oracle.pack(q), words)


def test_zero_point_pack_round_trip():
    rng = np.random.default_rng(3)
    z = rng.integers(0, 16, size=(32, 5), dtype=np.uint8)
    qz = oracle.pack_zeros(z)
    assert qz.shape == (4, 5)
    assert np.array_equal(oracle.unpack_zeros(qz, 32), z)
    assert np.array_equal(oracle.np_unpack_zeros(qz, 32), z)
    words = rng.integers(-2 ** 31, 2 ** 31, size=(4, 5), dtype=np.int64).astype(np.int32)
    assert np.array_equal(oracle.pack_zeros(oracle.unpack_zeros(words, 32)), words)


def test_nibble_order_single_elements():
    # element k = 8j + i lands in bits [4i, 4i+3] of word j
    for k in range(16):
        q = np.zeros((1, 16), dtype=np.uint8)
        q[0, k] = 0xF
        w = oracle.pack(q).astype(np.int64) & 0xFFFFFFFF
        expect = np.zeros(2, dtype=np.int64)
        expect[k // 8] = 0xF << (4 * (k % 8))
        assert np.array_equal(w[0], expect)
    for n in range(8):
        z = np.zeros((8, 1), dtype=np.uint8)
        z[n, 0] = 0xF
        w = int(oracle.pack_zeros(z)[0, 0]) & 0xFFFFFFFF
        assert w == 0xF << (4 * n)


# --------------------------------------------------------------------- golden
@pytest.mark.parametrize("name", CASES)
def test_hand_worked_cases(name):
    c = load(name)
    M, K, N, G, dt = c["M"], c["K"], c["N"], c["G"], c["dtype"]
    qw = oracle.pack(c["q"])
    if "qweight_words" in c:
        got = (qw.astype(np.int64) & 0xFFFFFFFF)[0].astype(np.uint64)
        assert np.array_equal(got, c["qweight_words"])
    s_bits = c["scales_bits"] if "scales_bits" in c else to_bits(c["scales_vals"], dt)
    qz = None
    if not c["sym"]:
        qz = oracle.pack_zeros(c["z"])
        assert (int(qz[0, 0]) & 0xFFFFFFFF) == int(c["qzeros_words"][0])
    x = to_bits(c["x_vals"], dt)
    if "w_bits" in c:
        w = oracle.dequant(qw, s_bits, qz, G, N, K, dt)
        assert np.array_equal(w[:, 0], c["w_bits"])
        assert np.all(w == w[:, :1])
    y = oracle.gemm(x, M, K, qw, s_bits, qz, G, N, dt)
    assert np.array_equal(y, c["y"]), (y, c["y"])
    if "y_exact" in c:
        ye = oracle.gemm(x, M, K, qw, s_bits, qz, G, N, dt, exact_weights=True)
        assert np.array_equal(ye, c["y_exact"])


# --------------------------------------------------------------------- identities
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_symmetric_equals_asymmetric_with_zero_point_8(dtype):
    p = make_problem(3, 16, 128, 32, True, dtype, seed=11)
    qw = oracle.pack(p.q)
    qz8 = oracle.pack_zeros(np.full((16, 4), 8, dtype=np.uint8))
    w_sym = oracle.dequant(qw, p.scales, None, 32, 16, 128, dtype)
    w_asym = oracle.dequant(qw, p.scales, qz8, 32, 16, 128, dtype)
    assert np.array_equal(w_sym, w_asym)
    y_sym = oracle.gemm(p.x, 3, 128, qw, p.scales, None, 32, 16, dtype)
    y_asym = oracle.gemm(p.x, 3, 128, qw, p.scales, qz8, 32, 16, dtype)
    assert np.array_equal(y_sym, y_asym)


def _np_dequant(p, dtype):
    """Numpy restatement: unpack by vector shifts, exact float64 product,
    library cast to the dtype."""
    qw = oracle.pack(p.q)
    q = oracle.np_unpack(qw, p.K).astype(np.int64)
    if p.z is None:
        z = np.full((p.N, p.n_groups), 8, dtype=np.int64)
    else:
        z = oracle.np_unpack_zeros(oracle.pack_zeros(p.z), p.N).astype(np.int64)
    if dtype == F16:
        s = p.scales.view(np.float16).astype(np.float64)
    else:
        s = (p.scales.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    zk = np.repeat(z, p.G, axis=1)
    sk = np.repeat(s, p.G, axis=1)
    prod = (q - zk).astype(np.float64) * sk
    if dtype == F16:
        return prod.astype(np.float16).astype(np.float64)
    return torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _x_vals(p, dtype):
    if dtype == F16:
        return p.x.view(np.float16).astype(np.float64)
    return (p.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("G", [32, 64])
def test_per_group_brute_force(sym, dtype, G):
    p = make_problem(2, 8, 128, G, sym, dtype, seed=5 + G)
    qw = oracle.pack(p.q)
    qz = None if sym else oracle.pack_zeros(p.z)
    w_np = _np_dequant(p, dtype)
    w_or = oracle.bits_to_float64(oracle.dequant(qw, p.scales, qz, G, 8, 128, dtype), dtype)
    assert np.array_equal(w_np, w_or)
    y_bf = oracle.np_gemm_bruteforce(_x_vals(p, dtype), w_np, G)
    y_or = oracle.gemm(p.x, 2, 128, qw, p.scales, qz, G, 8, dtype)
    np.testing.assert_allclose(y_or, y_bf, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_matches_float64_matmul(sym, dtype):
    p = make_problem(5, 64, 512, 128, sym, dtype, seed=21)
    qw = oracle.pack(p.q)
    qz = None if sym else oracle.pack_zeros(p.z)
    w = _np_dequant(p, dtype)
    y = oracle.gemm(p.x, 5, 512, qw, p.scales, qz, 128, 64, dtype)
    ref = _x_vals(p, dtype) @ w.T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-10)
    rows = np.array([4, 0, 2], dtype=np.int32)
    y_rows = oracle.gemm(p.x, 5, 512, qw, p.scales, qz, 128, 64, dtype, rows=rows)
    assert np.array_equal(y_rows, y[rows])


@pytest.mark.parametrize("sym", [True, False])
def test_integer_exact_gemm(sym):
    """s = 1 and integer x: every product and sum is an integer, so the oracle
    must equal an int64 matmul of (q - z) and x exactly."""
    M, N, K, G = 4, 16, 256, 64
    rng = np.random.default_rng(7)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    z = rng.integers(0, 16, size=(N, K // G), dtype=np.uint8)
    x = rng.integers(-4, 5, size=(M, K)).astype(np.int64)
    s_bits = np.full((N, K // G), 0x3C00, dtype=np.uint16)
    zz = np.full_like(z, 8) if sym else z
    qz = None if sym else oracle.pack_zeros(z)
    y = oracle.gemm(x.astype(np.float16).view(np.uint16), M, K, oracle.pack(q), s_bits, qz,
                    G, N, F16)
    w_int = q.astype(np.int64) - np.repeat(zz.astype(np.int64), G, axis=1)
    assert np.array_equal(y, (x @ w_int.T).astype(np.float64))


def test_rows_subset_and_exact_weights_flag():
    p = make_problem(3, 8, 64, 32, False, BF16, seed=9)
    qw, qz = oracle.pack(p.q), oracle.pack_zeros(p.z)
    y = oracle.gemm(p.x, 3, 64, qw, p.scales, qz, 32, 8, BF16)
    ye = oracle.gemm(p.x, 3, 64, qw, p.scales, qz, 32, 8, BF16, exact_weights=True)
    assert not np.array_equal(y, ye)           # bf16 weight rounding is visible
    np.testing.assert_allclose(y, ye, rtol=0.05, atol=0.05)


# --------------------------------------------------------------------- fused epilogue
def test_epilogue_bias_closed_forms():
    """With x = 0 the layer output is the bias itself (exact values of its
    bit patterns); adding a bias shifts every row by the same vector."""
    p = make_problem(3, 16, 64, 32, False, F16, seed=41)
    bias = np.array([0x3C00, 0xBC00, 0x3800, 0x0001, 0x7BFF, 0, 0x8000, 0x4248] * 2, dtype=np.uint16)
    zero_x = np.zeros_like(p.x)
    qw = oracle.pack(p.q)
    qz = oracle.pack_zeros(p.z)
    y0 = oracle.gemm(zero_x, 3, 64, qw, p.scales, qz, 32, 16, F16)
    a0 = oracle.epilogue(y0, 16, F16, bias=bias)
    want = bias.view(np.float16).astype(np.float64)
    assert np.array_equal(a0, np.tile(want, (3, 1)))
    y = oracle.gemm(p.x, 3, 64, qw, p.scales, qz, 32, 16, F16)
    a = oracle.epilogue(y, 16, F16, bias=bias)
    np.testing.assert_allclose(a - y, np.tile(want, (3, 1)), rtol=0, atol=1e-12 * (1 + np.abs(y).max()))
    assert np.array_equal(oracle.epilogue(y, 16, F16), y)


def test_epilogue_silu_special_values():
    """sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4, so silu(+-ln 3) =
    +-(3/4 or -1/4) ln 3; silu(0) = 0; silu(v) - silu(-v) = v for every v
    (sigmoid(v) + sigmoid(-v) = 1); the up half multiplies column by column."""
    l3 = np.log(3.0)
    y = np.array([[0.0, l3, -l3, 2.0, 1.0, 3.0]])
    h = oracle.epilogue(y, 6, BF16, silu_mul=True)
    np.testing.assert_allclose(h[0], [0.0, 0.75 * l3 * 1.0, -0.25 * l3 * 3.0], rtol=1e-15, atol=0)
    v = np.linspace(-30, 30, 241)
    ypos = np.concatenate([v, np.ones_like(v)])[None, :]
    yneg = np.concatenate([-v, np.ones_like(v)])[None, :]
    d = oracle.epilogue(ypos, 482, F16, silu_mul=True) - oracle.epilogue(yneg, 482, F16, silu_mul=True)
    np.testing.assert_allclose(d[0], v, rtol=0, atol=1e-13)


def test_epilogue_silu_mul_against_torch():
    """The whole epilogue on a real layer's accumulations against torch's
    SiLU (its own implementation) on the gate half times the up half, with
    the bias of each half added first."""
    p = make_problem(4, 64, 128, 64, True, BF16, seed=43)
    qw = oracle.pack(p.q)
    y = oracle.gemm(p.x, 4, 128, qw, p.scales, None, 64, 64, BF16)
    rng = np.random.default_rng(5)
    bias_f = rng.uniform(-2, 2, 64).astype(np.float32)
    bias = torch.from_numpy(bias_f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bv = bias.astype(np.uint32) << 16
    b64 = bv.view(np.float32).astype(np.float64)
    h = oracle.epilogue(y, 64, BF16, bias=bias, silu_mul=True)
    a = torch.from_numpy(y + b64)
    want = torch.nn.functional.silu(a[:, :32]) * a[:, 32:]
    np.testing.assert_allclose(h, want.numpy(), rtol=1e-12, atol=1e-12)
    # the halves are not interchangeable: swapping them changes the result
    swapped = torch.nn.functional.silu(a[:, 32:]) * a[:, :32]
    assert not np.allclose(h, swapped.numpy())


# --------------------------------------------------------------------- MoE
def _experts(E, N, K, G, sym, dtype, seed):
    ps = [make_problem(1, N, K, G, sym, dtype, seed=seed + e) for e in range(E)]
    qw = np.stack([oracle.pack(p.q) for p in ps])
    sc = np.stack([p.scales for p in ps])
    qz = None if sym else np.stack([oracle.pack_zeros(p.z) for p in ps])
    return ps, qw, sc, qz


def test_moe_single_expert_is_the_gemm():
    """One expert, every token routed to it: the MoE result is the plain
    GEMM of all tokens (the pinned routine), row for row."""
    ps, qw, sc, qz = _experts(1, 16, 64, 32, False, F16, 51)
    x = make_problem(3, 16, 64, 32, False, F16, seed=52).x
    got = oracle.moe_gemm(x, 3, 64, qw, sc, qz, 32, 16, np.zeros((3, 2), np.int32), F16)
    want = oracle.gemm(x, 3, 64, qw[0], sc[0], qz[0], 32, 16, F16)
    assert np.array_equal(got[:, 0], want) and np.array_equal(got[:, 1], want)


def test_moe_brute_force_and_routing():
    """Against a numpy restatement (unpack, RN of (q - z) s through torch,
    float64 dot products) on routed tokens with repeated experts and routing
    weights; relabelling the experts (permuting the weight stack and the ids
    alike) changes nothing."""
    E, N, K, G = 4, 8, 64, 32
    ps, qw, sc, qz = _experts(E, N, K, G, False, BF16, 61)
    x = make_problem(3, N, K, G, False, BF16, seed=62).x
    ids = np.array([[2, 0], [1, 1], [3, 2]], dtype=np.int32)
    rw = np.array([[0.25, 0.75], [1.0, -0.5], [2.0, 0.125]])
    got = oracle.moe_gemm(x, 3, K, qw, sc, qz, G, N, ids, BF16, route_weights=rw)
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(3):
        for j in range(2):
            p = ps[ids[t, j]]
            q = p.q.astype(np.int64)
            z = np.repeat(p.z.astype(np.int64), G, axis=1)
            s = (np.repeat(p.scales, G, axis=1).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            wv = torch.from_numpy((q - z) * s).to(torch.bfloat16).to(torch.float64).numpy()
            np.testing.assert_allclose(got[t, j], (wv @ xv[t]) * rw[t, j], rtol=1e-12, atol=1e-12)
    perm = np.array([3, 1, 0, 2])                 # new expert i is old expert perm[i]
    inv = np.argsort(perm)
    got2 = oracle.moe_gemm(x, 3, K, qw[perm], sc[perm], qz[perm], G, N, inv[ids], BF16, route_weights=rw)
    assert np.array_equal(got, got2)
