"""Pins for the CPU oracle: each test checks it against something other than
itself (hand-packed fixtures, exact rational arithmetic, the definition of
ties-to-even, identities of the method, a library matmul).

Sources: Predibase Lorax "AWQ WQLinear" page -- I/O Contract (qweight int32
[in_features, out_features // 8], packed qzeros, per-group scales, optional
bias), Description (__init__ shape rules and group_size -1; forward: flatten,
quantised GEMM, bias). The nibble order, the qzeros/scales shapes and the
fp16 rounding of dequantised weights are the library's fixed readings.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bit_weight_quantized_awq_gb300.synthetic import make_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_fixture(name):
    with open(os.path.join(GOLDEN, name)) as f:
        d = json.load(f)
    d["qweight"] = np.array([[int(w, 16) for w in row] for row in d["qweight_hex"]],
                            dtype=np.uint32).view(np.int32)
    d["qzeros"] = np.array([[int(w, 16) for w in row] for row in d["qzeros_hex"]],
                           dtype=np.uint32).view(np.int32)
    d["q"] = np.array([[int(c, 16) for c in s] for s in d["q_rows"]], dtype=np.int64)
    d["z"] = np.array([[int(c, 16) for c in s] for s in d["z_rows"]], dtype=np.int64)
    return d


def _np16(values):
    return np.asarray(values, dtype=np.float64).astype(np.float16)


# --------------------------------------------------------------------------
# binary16 conversions
# --------------------------------------------------------------------------

ALL16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_f16_decode_every_pattern_matches_numpy():
    mine = oracle.f16_bits_to_f64(ALL16)
    ref = ALL16.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # sign of zero survives
    assert np.signbit(mine[0x8000]) and not np.signbit(mine[0x0000])


def test_f16_roundtrip_every_finite_pattern():
    finite = ALL16[(ALL16 & 0x7C00) != 0x7C00]
    back = oracle.f64_to_f16_bits(oracle.f16_bits_to_f64(finite))
    assert np.array_equal(back, finite)
    inf = np.array([0x7C00, 0xFC00], dtype=np.uint16)
    assert np.array_equal(oracle.f64_to_f16_bits(oracle.f16_bits_to_f64(inf)), inf)
    assert (oracle.f64_to_f16_bits(np.array([np.nan]))[0] & 0x7C00) == 0x7C00


def _neighbours():
    """Every pair of adjacent non-negative finite binary16 values (a, b) as
    bit patterns, a < b, plus the pair (65504, overflow)."""
    lo = np.arange(0, 0x7BFF, dtype=np.uint32).astype(np.uint16)
    return lo, (lo + 1).astype(np.uint16)


def test_f16_encode_ties_go_to_even_fraction():
    a, b = _neighbours()
    fa, fb = a.view(np.float16).astype(np.float64), b.view(np.float16).astype(np.float64)
    mid = (fa + fb) / 2  # exact in binary64
    # ties-to-even, from the definition: the neighbour whose last fraction bit is 0
    expect = np.where((a & 1) == 0, a, b)
    assert np.array_equal(oracle.f64_to_f16_bits(mid), expect)
    assert np.array_equal(oracle.f64_to_f16_bits(-mid), expect | 0x8000)
    # just off the midpoint, the nearer neighbour wins
    up = np.nextafter(mid, np.inf)
    dn = np.nextafter(mid, -np.inf)
    assert np.array_equal(oracle.f64_to_f16_bits(up), b)
    assert np.array_equal(oracle.f64_to_f16_bits(dn), a)


def test_f16_encode_overflow_and_underflow_edges():
    cases = {
        65504.0: 0x7BFF,
        65519.99: 0x7BFF,
        65520.0: 0x7C00,          # tie between 65504 and 2^16: even side overflows
        1e9: 0x7C00,
        2.0 ** -24: 0x0001,       # smallest subnormal
        2.0 ** -25: 0x0000,       # tie between 0 and 2^-24 -> even (0)
        3 * 2.0 ** -25: 0x0002,   # tie between 1 and 2 ulps -> even (2)
        np.nextafter(2.0 ** -25, 1): 0x0001,
        2.0 ** -14: 0x0400,       # smallest normal
        (2.0 ** -14) * (1 - 2.0 ** -11): 0x0400,  # tie between largest subnormal and min normal -> even
    }
    for v, bits in cases.items():
        assert int(oracle.f64_to_f16_bits(np.array([v]))[0]) == bits, v
        assert int(oracle.f64_to_f16_bits(np.array([-v]))[0]) == bits | 0x8000, -v


def test_f16_encode_random_matches_numpy():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(200_000) * np.exp2(rng.integers(-30, 18, 200_000))
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f64_to_f16_bits(v), ref)


# --------------------------------------------------------------------------
# shape rules
# --------------------------------------------------------------------------

def test_group_rules():
    assert oracle.resolve_group(4096, 4096, -1) == 4096
    assert oracle.resolve_group(4096, 4096, 128) == 128
    assert oracle.resolve_group(4096, 8, 4096) == 4096
    assert oracle.resolve_group(4096, 12, 128) is None      # N % 8 != 0
    assert oracle.resolve_group(4096, 4096, 100) is None    # K % g != 0
    assert oracle.resolve_group(4096, 4096, 0) is None
    assert oracle.resolve_group(4096, 4096, -2) is None
    assert oracle.resolve_group(0, 8, -1) is None


# --------------------------------------------------------------------------
# unpack: hand-packed fixtures and one-hot placement
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["hand_8x8.json", "hand_16x16.json"])
def test_unpack_hand_packed(name):
    d = _load_fixture(name)
    assert np.array_equal(oracle.unpack(d["qweight"]), d["q"])
    assert np.array_equal(oracle.unpack(d["qzeros"]), d["z"])


def test_unpack_literal_words():
    words = np.array([[0x76543210, 0xFEDCBA98], [0x0000000F, 0xF0000000]],
                     dtype=np.uint32).view(np.int32)
    codes = oracle.unpack(words)
    assert codes[0].tolist() == list(range(16))
    assert codes[1].tolist() == [15] + [0] * 14 + [15]


@pytest.mark.parametrize("k0", [0, 5, 15])
def test_one_hot_places_each_nibble_slot(k0):
    """q == z everywhere except q[k0, c0] = z + 1, scale 1: W is a single 1.0
    at (k0, c0), so y[:, c0] == x[:, k0] and every other column is zero."""
    K, N, M = 16, 16, 3
    x = make_problem(M, K, N, K).x.numpy()
    zword = 0x55555555
    qzeros = np.full((1, N // 8), zword, dtype=np.uint32).view(np.int32)
    scales = np.ones((1, N), dtype=np.float16)
    xs = x.astype(np.float64)
    for c0 in range(N):
        qw = np.full((K, N // 8), zword, dtype=np.uint32)
        qw[k0, c0 // 8] = zword + (1 << (4 * (c0 % 8)))   # that one code becomes 6
        y = oracle.forward(x, qw.view(np.int32), qzeros, scales, None, K)
        expect = np.zeros((M, N))
        expect[:, c0] = xs[:, k0]
        assert np.array_equal(y, expect), c0


# --------------------------------------------------------------------------
# dequant: exhaustive (q, z) x every finite fp16 scale
# --------------------------------------------------------------------------

def test_dequant_exhaustive_q_z_and_scales():
    """Row k has every code = k; column 16b + z has zero point z and scale
    s_b. Expected W16 = numpy's correctly rounded fp16 of the exact product."""
    finite = ALL16[(ALL16 & 0x7C00) != 0x7C00]
    S = finite.size
    K, N = 16, 16 * S
    qweight = (np.arange(16, dtype=np.uint32)[:, None] * np.uint32(0x11111111)
               * np.ones((1, N // 8), dtype=np.uint32)).view(np.int32)
    zrow = np.tile(np.array([0x76543210, 0xFEDCBA98], dtype=np.uint32), S)[None, :]
    qzeros = zrow.view(np.int32)
    scales = np.repeat(finite, 16)[None, :]
    W16 = oracle.dequant(qweight, qzeros, scales, 16)
    q = np.arange(16, dtype=np.float64)[:, None]
    z = np.tile(np.arange(16, dtype=np.float64), S)[None, :]
    s = scales.view(np.float16).astype(np.float64)
    with np.errstate(over="ignore"):
        expect = ((q - z) * s).astype(np.float16).view(np.uint16)   # product exact in fp64
    assert np.array_equal(W16, expect)


@pytest.mark.parametrize("name", ["hand_8x8.json", "hand_16x16.json"])
def test_dequant_and_forward_hand_cases_exact(name):
    """Brute force in exact rationals; every value is a small dyadic, so the
    fp16 weights and the fp64 sums are exact and must match bit for bit."""
    d = _load_fixture(name)
    M, K, N, gs = d["M"], d["K"], d["N"], d["group_size"]
    g = K if gs == -1 else gs
    scales = _np16(d["scales"])
    x = _np16(d["x"])
    bias = None if d["bias"] is None else _np16(d["bias"])
    W = [[Fraction(int(d["q"][k][n]) - int(d["z"][k // g][n])) * Fraction(d["scales"][k // g][n])
          for n in range(N)] for k in range(K)]
    W16 = oracle.dequant(d["qweight"], d["qzeros"], scales, gs)
    assert np.array_equal(oracle.f16_bits_to_f64(W16), np.array([[float(w) for w in r] for r in W]))
    y = oracle.forward(x, d["qweight"], d["qzeros"], scales, bias, gs)
    for m in range(M):
        for n in range(N):
            acc = sum(Fraction(d["x"][m][k]) * W[k][n] for k in range(K))
            if d["bias"] is not None:
                acc += Fraction(d["bias"][n])
            assert y[m, n] == float(acc), (m, n)


# --------------------------------------------------------------------------
# identities of the method on seeded inputs
# --------------------------------------------------------------------------

def _np(p):
    return (p.x.numpy(), p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(),
            None if p.bias is None else p.bias.numpy())


@pytest.mark.parametrize("with_bias", [True, False])
def test_q_equal_z_gives_bias(with_bias):
    M, K, N, g = 4, 256, 64, 64
    p = make_problem(M, K, N, g, bias=with_bias, seed=3)
    x, _, qz, sc, b = _np(p)
    qw = np.repeat(qz, g, axis=0)             # every code equals its zero point
    sc = sc.copy()
    sc[:, ::2] = -sc[:, ::2]                  # negative scales give -0.0 weights
    W16 = oracle.dequant(qw, qz, sc, g)
    assert np.array_equal(W16, np.where(np.repeat(sc.view(np.uint16) & 0x8000, g, axis=0) != 0,
                                        0x8000, 0x0000).astype(np.uint16))
    y = oracle.forward(x, qw, qz, sc, b, g)
    expect = np.zeros((M, N)) if b is None else np.broadcast_to(b.astype(np.float64), (M, N))
    assert np.array_equal(y, expect)


def test_group_minus_one_equals_group_k():
    p = make_problem(3, 512, 128, -1, bias=True, seed=4)
    x, qw, qz, sc, b = _np(p)
    assert np.array_equal(oracle.forward(x, qw, qz, sc, b, -1),
                          oracle.forward(x, qw, qz, sc, b, 512))
    assert np.array_equal(oracle.dequant(qw, qz, sc, -1), oracle.dequant(qw, qz, sc, 512))


def test_doubling_scales_doubles_y():
    p = make_problem(5, 384, 96, 128, bias=False, seed=5)
    x, qw, qz, sc, _ = _np(p)
    sc2 = (sc.astype(np.float64) * 2).astype(np.float16)
    y1 = oracle.forward(x, qw, qz, sc, None, 128)
    y2 = oracle.forward(x, qw, qz, sc2, None, 128)
    assert np.array_equal(y2, 2 * y1)


def test_sum_of_per_group_partial_products():
    """A wrong group index (k % g instead of k // g, or a transposed scale
    table) breaks this: y equals the sum over groups of the matmul restricted
    to that group's input rows with that group's zeros and scales."""
    M, K, N, g = 3, 512, 64, 128
    p = make_problem(M, K, N, g, bias=False, seed=6)
    x, qw, qz, sc, _ = _np(p)
    total = np.zeros((M, N))
    for gi in range(K // g):
        ks = slice(gi * g, (gi + 1) * g)
        total += oracle.forward(np.ascontiguousarray(x[:, ks]), qw[ks], qz[gi:gi + 1],
                                sc[gi:gi + 1], None, g)
    y = oracle.forward(x, qw, qz, sc, None, g)
    np.testing.assert_allclose(y, total, rtol=1e-12, atol=1e-12)


def test_forward_matches_library_matmul():
    """Library cross-check: oracle W16 -> numpy fp64 matmul + bias."""
    p = make_problem(7, 640, 136, 128, bias=True, seed=7)
    x, qw, qz, sc, b = _np(p)
    W = oracle.f16_bits_to_f64(oracle.dequant(qw, qz, sc, 128))
    ref = x.astype(np.float64) @ W + b.astype(np.float64)
    y = oracle.forward(x, qw, qz, sc, b, 128)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_row_sample_and_threads_do_not_change_values():
    p = make_problem(9, 256, 64, 64, bias=True, seed=8)
    x, qw, qz, sc, b = _np(p)
    full1 = oracle.forward(x, qw, qz, sc, b, 64, threads=1)
    full8 = oracle.forward(x, qw, qz, sc, b, 64, threads=8)
    assert np.array_equal(full1, full8)
    rows = [8, 0, 3]
    assert np.array_equal(oracle.forward(x, qw, qz, sc, b, 64, rows=rows), full1[rows])


def test_three_d_input_is_flattened():
    """Forward step 1 on the WQLinear page: x [..., K] is reshaped to 2-D."""
    p = make_problem(2 * 3, 64, 16, -1, bias=True, seed=9, x_shape=(2, 3, 64))
    x, qw, qz, sc, b = _np(p)
    y3 = oracle.forward(x, qw, qz, sc, b, -1)
    y2 = oracle.forward(x.reshape(6, 64), qw, qz, sc, b, -1)
    assert np.array_equal(y3, y2)


# --------------------------------------------------------------------------
# pack (the inverse of unpack): hand-packed fixtures, closed form, round trips
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["hand_8x8.json", "hand_16x16.json"])
def test_pack_hand_packed(name):
    d = _load_fixture(name)
    assert np.array_equal(oracle.pack(d["q"].astype(np.uint8)), d["qweight"])
    assert np.array_equal(oracle.pack(d["z"].astype(np.uint8)), d["qzeros"])


def test_pack_one_hot_closed_form():
    """Code v at column c of a row is v << 4 (c mod 8) in word c // 8."""
    for c in range(16):
        for v in (1, 7, 15):
            codes = np.zeros((2, 16), dtype=np.uint8)
            codes[1, c] = v
            expect = np.zeros((2, 2), dtype=np.uint32)
            expect[1, c // 8] = v << (4 * (c % 8))
            assert np.array_equal(oracle.pack(codes).view(np.uint32), expect), (c, v)


def test_pack_and_unpack_round_trips():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, size=(37, 96), dtype=np.uint8)
    assert np.array_equal(oracle.unpack(oracle.pack(codes)), codes)
    words = rng.integers(0, 2**32, size=(11, 5), dtype=np.uint64).astype(np.uint32).view(np.int32)
    assert np.array_equal(oracle.pack(oracle.unpack(words)), words)
    # only the low four bits of a code are used
    assert np.array_equal(oracle.pack(codes | np.uint8(0xF0)), oracle.pack(codes))


# --------------------------------------------------------------------------
# round-to-nearest quantisation: q = clamp(round_half_even(W / s) + z, 0, 15)
# --------------------------------------------------------------------------

def test_quantize_recovers_codes_on_exact_grid_points():
    """Power-of-two scales make W = (q - z) s exact in fp16: q comes back."""
    rng = np.random.default_rng(4)
    K, N, g = 64, 48, 16
    G = K // g
    q = rng.integers(0, 16, size=(K, N))
    z = rng.integers(0, 16, size=(G, N))
    s = np.ldexp(1.0, rng.integers(-10, 2, size=(G, N))).astype(np.float16)
    Wx = (q - np.repeat(z, g, axis=0)) * np.repeat(s.astype(np.float64), g, axis=0)
    W = Wx.astype(np.float16)
    assert np.array_equal(W.astype(np.float64), Wx)   # every point is exact in fp16
    got = oracle.unpack(oracle.quantize_rtn(W, s, oracle.pack(z.astype(np.uint8)), g))
    assert np.array_equal(got, q)


def test_quantize_hand_cases_ties_and_clamping():
    """W / s on halves (ties to the even integer), just off halves, and far
    outside the code range; zero point 8. Expected codes worked by hand from
    clamp(round_half_even(t) + 8, 0, 15)."""
    t = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.375, 3.625, 100.0, -100.0, 7.5, -8.5, 0.0, 6.5, -7.5, -6.5]
    expect = [8, 10, 10, 8, 6, 6, 11, 12, 15, 0, 15, 0, 8, 14, 0, 2]
    N = len(t)
    s = np.full((1, N), 0.25, dtype=np.float16)
    W = (np.array(t) * 0.25).astype(np.float16).reshape(1, N)
    assert np.array_equal(W.astype(np.float64).ravel(), np.array(t) * 0.25)
    z = np.full((1, N), 8, dtype=np.uint8)
    got = oracle.unpack(oracle.quantize_rtn(W, s, oracle.pack(z), -1))
    assert got.ravel().tolist() == expect


def test_quantize_zero_and_infinite_quotients():
    """s = 0: 0 / 0 counts as 0 (code = z); x / 0 is infinite and clamps."""
    W = np.array([[0.0, 1.0, -1.0, 0.0, 0.0, 0.0, 0.0, 0.0]], dtype=np.float16)
    s = np.array([[0.0, 0.0, 0.0, 1.0, 1.0, 1.0, 1.0, 1.0]], dtype=np.float16)
    z = np.array([[5, 5, 5, 0, 15, 3, 3, 3]], dtype=np.uint8)
    got = oracle.unpack(oracle.quantize_rtn(W, s, oracle.pack(z), 1))
    assert got.ravel().tolist() == [5, 15, 0, 0, 15, 3, 3, 3]


@pytest.mark.parametrize("K,N,g", [(256, 64, 32), (128, 40, -1), (96, 16, 48)])
def test_quantize_inverts_dequant_for_any_scale(K, N, g):
    """|fp16_rn((q - z) s) / s - (q - z)| <= 15 * 2^-11 < 1/2, so rounding the
    quotient gives q - z back: quantize(dequant(q)) == q for normal scales."""
    p = make_problem(1, K, N, g, seed=K + N)
    W = oracle.dequant(p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), g)
    back = oracle.quantize_rtn(W, p.scales.numpy(), p.qzeros.numpy(), g)
    assert np.array_equal(back, p.qweight.numpy())


# --------------------------------------------------------------------------
# grouping by table (g_idx): the group of input row k is g_idx[k]
# --------------------------------------------------------------------------

@pytest.mark.parametrize("K,N,g", [(256, 64, 32), (96, 16, 48), (64, 40, -1)])
def test_gidx_with_floor_table_equals_grouped(K, N, g):
    """g_idx[k] = k // g reproduces the grouped dequant and forward exactly."""
    p = make_problem(5, K, N, g, bias=True, seed=K + 1)
    gg = K if g == -1 else g
    table = (np.arange(K) // gg).astype(np.int32)
    qw, qz, sc = p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy()
    assert np.array_equal(oracle.dequant_gidx(qw, qz, sc, table), oracle.dequant(qw, qz, sc, g))
    y1 = oracle.forward_gidx(p.x.numpy(), qw, qz, sc, table, p.bias.numpy())
    y2 = oracle.forward(p.x.numpy(), qw, qz, sc, p.bias.numpy(), g)
    assert np.array_equal(y1, y2)


def test_gidx_follows_a_permutation_of_the_rows():
    """Permuting the rows of qweight together with g_idx permutes the rows of
    W16; permuting x's columns the same way leaves y unchanged."""
    K, N, G = 96, 32, 6
    p = make_problem(3, K, N, K // G * 1, bias=False, seed=7)
    rng = np.random.default_rng(11)
    table = rng.integers(0, G, size=K).astype(np.int32)
    qw, qz, sc = p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy()
    assert qz.shape[0] == G
    perm = rng.permutation(K)
    W = oracle.dequant_gidx(qw, qz, sc, table)
    Wp = oracle.dequant_gidx(np.ascontiguousarray(qw[perm]), qz, sc, table[perm])
    assert np.array_equal(Wp, W[perm])
    x = p.x.numpy()
    y = oracle.forward_gidx(x, qw, qz, sc, table, None)
    yp = oracle.forward_gidx(np.ascontiguousarray(x[:, perm]), np.ascontiguousarray(qw[perm]), qz, sc,
                             table[perm], None)
    assert np.allclose(yp, y, rtol=1e-12, atol=1e-12)


def test_gidx_constant_table_is_one_group():
    """Every row in group c: the dequant of a single group (g = K) with group
    c's scales and zero points."""
    K, N, G = 64, 24, 4
    p = make_problem(1, K, N, K // G, seed=13)
    qw, qz, sc = p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy()
    for c in range(G):
        table = np.full(K, c, dtype=np.int32)
        expect = oracle.dequant(qw, np.ascontiguousarray(qz[c:c + 1]), np.ascontiguousarray(sc[c:c + 1]), -1)
        assert np.array_equal(oracle.dequant_gidx(qw, qz, sc, table), expect), c


def test_gidx_rejects_out_of_range_groups():
    p = make_problem(1, 32, 16, 8, seed=3)
    table = np.zeros(32, dtype=np.int32)
    table[5] = 4                      # G = 4 groups: 0..3
    with pytest.raises(ValueError):
        oracle.dequant_gidx(p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), table)
    table[5] = -1
    with pytest.raises(ValueError):
        oracle.dequant_gidx(p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), table)
