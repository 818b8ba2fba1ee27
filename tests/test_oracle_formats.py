"""Pins of the oracle's number formats against what the formats themselves fix.

fp16 against the IEEE-754 definition and numpy's independent conversion;
Q4_K / Q4_0 unpacking against hand-built blocks (tests/golden); Q8_1
quantisation against closed forms on grid inputs.  No expected value here comes
from the oracle or from the CUDA path.
"""
import json
import os

import numpy as np
import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden", "handbuilt_blocks.json")


@pytest.fixture(scope="module")
def gold():
    with open(GOLD) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- fp16
def test_f16_exhaustive_roundtrip(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (h >> 10) & 31
    frac = h & 1023
    finite_or_inf = ~((exp == 31) & (frac != 0))
    vals = np.frombuffer(h.tobytes(), np.float16).astype(np.float32)
    back = orc.f32_to_f16(vals)
    assert np.array_equal(back[finite_or_inf], h[finite_or_inf])
    # NaNs stay NaN
    nan_back = back[~finite_or_inf]
    assert np.all(((nan_back >> 10) & 31) == 31) and np.all((nan_back & 1023) != 0)


def test_f16_to_f64_definition(orc):
    # value = 2^(e-15) * (1 + f/1024), subnormal 2^-14 * f/1024
    cases = {0x3C00: 1.0, 0x3800: 0.5, 0x4000: 2.0, 0xC000: -2.0, 0x7BFF: 65504.0,
             0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24, 0x0400: 2.0 ** -14,
             0x3555: 1.0 / 4 * (1 + 0x155 / 1024), 0x8000: -0.0}
    got = orc.f16_to_f64(np.array(list(cases), np.uint16))
    assert np.array_equal(got, np.array(list(cases.values())))
    assert np.isinf(orc.f16_to_f64(np.array([0x7C00], np.uint16)))[0]


def test_f32_to_f16_matches_numpy_random(orc):
    g = np.random.default_rng(1234)
    bits = g.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    # concentrate on the interesting range too: normals, subnormals, overflow edge
    y = np.concatenate([x, g.uniform(-70000, 70000, 100_000).astype(np.float32),
                        (g.standard_normal(100_000) * 1e-5).astype(np.float32),
                        (g.standard_normal(100_000) * 1e-7).astype(np.float32)])
    ours = orc.f32_to_f16(y)
    with np.errstate(over="ignore"):
        ref = y.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("x,bits", [
    (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00), (1e9, 0x7C00),
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (3 * 2.0 ** -25, 0x0002),
    (1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02), (-1.0, 0xBC00),
    (2.0 ** -14 - 2.0 ** -25, 0x0400),
])
def test_f32_to_f16_ties_and_edges(orc, x, bits):
    assert int(orc.f32_to_f16(np.array([x], np.float32))[0]) == bits


# ----------------------------------------------------------------------------- Q4_K
def _block_with(scale_bytes, d_bits=0x3C00, dmin_bits=0x3800, qs=None):
    b = np.zeros(144, np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    b[2], b[3] = dmin_bits & 0xFF, dmin_bits >> 8
    b[4:16] = scale_bytes
    if qs is not None:
        b[16:] = qs
    return b


def test_q4k_scale_unpack_handbuilt(orc, gold):
    g = gold["q4k_scales"]
    d, dm, sc, mn, q = orc.q4k_unpack(_block_with(g["scale_bytes"]))
    assert (d, dm) == (0x3C00, 0x3800)
    assert sc.tolist() == g["sc"]
    assert mn.tolist() == g["m"]


def test_q4k_nibble_unpack_handbuilt(orc, gold):
    for case in gold["q4k_nibbles"]["cases"]:
        qs = np.zeros(128, np.uint8)
        qs[case["k"]] = 0xB7
        _, _, _, _, q = orc.q4k_unpack(_block_with(np.zeros(12, np.uint8), qs=qs))
        expect = np.zeros(256, np.uint8)
        expect[case["low_element"]] = 7
        expect[case["high_element"]] = 11
        assert np.array_equal(q, expect), case


def test_q4k_dequant_handbuilt(orc, gold):
    g = gold["q4k_dequant"]
    qs = np.zeros(128, np.uint8)
    qs[g["k"]] = g["byte"]
    blk = _block_with(gold["q4k_scales"]["scale_bytes"], g["d_bits"], g["dmin_bits"], qs)
    w = orc.q4k_dequantize(blk[None, :])[0]
    for e, v in g["expect"].items():
        assert w[int(e)] == v, (e, w[int(e)], v)


def test_q4k_pack_unpack_roundtrip(orc):
    g = np.random.default_rng(7)
    for trial in range(200):
        sc = g.integers(0, 64, 8).astype(np.uint8)
        mn = g.integers(0, 64, 8).astype(np.uint8)
        if trial < 5:   # corner values 0, 1, 31, 32, 63
            sc[:] = [0, 1, 31, 32, 63, 63, 0, 32][trial:] + [0, 1, 31, 32, 63, 63, 0, 32][:trial]
        q = g.integers(0, 16, 256).astype(np.uint8)
        d, dm = int(g.integers(0, 0x7C00)), int(g.integers(0, 0x7C00))
        blk = orc.q4k_pack(d, dm, sc, mn, q)
        d2, dm2, sc2, mn2, q2 = orc.q4k_unpack(blk)
        assert (d2, dm2) == (d, dm)
        assert np.array_equal(sc2, sc) and np.array_equal(mn2, mn) and np.array_equal(q2, q)
    # every one of the 2^(12*8) scale patterns is reachable: unpack(pack(unpack(b))) == b
    for _ in range(200):
        blk = g.integers(0, 256, 144).astype(np.uint8)
        again = orc.q4k_pack(*orc.q4k_unpack(blk))
        assert np.array_equal(again, blk)


# ----------------------------------------------------------------------------- Q4_0
def test_q4_0_handbuilt(orc, gold):
    g = gold["q4_0"]
    blk = np.zeros(18, np.uint8)
    blk[0], blk[1] = g["d_bits"] & 0xFF, g["d_bits"] >> 8
    blk[2 + g["k"]] = g["byte"]
    w = orc.q4_0_dequantize(blk[None, :])[0]
    for e, v in g["expect"].items():
        assert w[int(e)] == v
    d, q = orc.q4_0_unpack(blk)
    assert np.array_equal(orc.q4_0_pack(d, q), blk)


# ----------------------------------------------------------------------------- Q8_1
def test_q8_1_grid_inputs_recover_integers(orc):
    """x_i = k_i * c with max|k| = 127 quantises to q_i = k_i exactly."""
    g = np.random.default_rng(3)
    for c in [0.125, 1.0, 3.7e-3, 17.25, 1e-4]:
        k = g.integers(-127, 128, (8, 32))
        k[:, 5] = 127 * np.where(g.random(8) < 0.5, 1, -1)   # pin amax
        x = (k * c).astype(np.float32)
        q8 = orc.q8_1_quantize(x.reshape(1, -1))
        d, s, q = orc.q8_1_fields(q8, 1, 256)
        assert np.array_equal(q[0].astype(np.int64), k)
        # d is the f32 quotient max|x| / 127
        expect_d = np.float32(np.float32(127 * c) / np.float32(127))
        assert np.array_equal(d[0], np.full(8, expect_d, np.float32))
        # s is the f32 product d * sum(q)
        assert np.array_equal(s[0], (d[0] * k.sum(axis=1).astype(np.float32)).astype(np.float32))
        if c == 0.125:   # everything exact
            assert np.array_equal(s[0].astype(np.float64), 0.125 * k.sum(axis=1))


def test_q8_1_zero_and_one_hot(orc):
    x = np.zeros((1, 64), np.float32)
    x[0, 32 + 9] = -3.5
    d, s, q = orc.q8_1_fields(orc.q8_1_quantize(x), 1, 64)
    assert d[0, 0] == 0 and s[0, 0] == 0 and not q[0, 0].any()
    assert q[0, 1, 9] == -127 and np.count_nonzero(q[0, 1]) == 1
    assert d[0, 1] == np.float32(3.5) / np.float32(127)
    assert s[0, 1] == d[0, 1] * np.float32(-127)


def test_q8_1_rounding_half_away_from_zero(orc):
    """With amax = 127, d = 1 exactly and q = round(x): ties go away from zero."""
    x = np.zeros((1, 32), np.float32)
    x[0, :8] = [127, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 0.49999997]
    _, _, q = orc.q8_1_fields(orc.q8_1_quantize(x), 1, 32)
    assert q[0, 0, :8].tolist() == [127, 1, 2, 3, -1, -2, -3, 0]


def test_q8_1_large_block_sum_stays_finite(orc):
    """Activations of order 1e5 (the size the random Llama-shaped FFN reaches): the
    sum term s = d * sum(q) is finite (an fp16 s would overflow above 65504)."""
    x = np.full((1, 32), 9.0e4, np.float32)
    d, s, q = orc.q8_1_fields(orc.q8_1_quantize(x), 1, 32)
    assert np.all(q == 127) and np.isfinite(s[0, 0])
    assert abs(float(s[0, 0]) - 32 * 9.0e4) <= 32 * 9.0e4 * 2 ** -22


def test_q8_1_blocks_independent_and_bounded(orc):
    g = np.random.default_rng(5)
    x = g.standard_normal((3, 256)).astype(np.float32)
    q8 = orc.q8_1_quantize(x)
    d, s, q = orc.q8_1_fields(q8, 3, 256)
    assert np.all(np.abs(q.astype(int)) <= 127)
    assert np.all(np.abs(q.astype(int)).max(axis=-1) == 127)
    # perturbing one block changes only that block
    x2 = x.copy()
    x2[1, 40] *= 2
    d2, s2, q2 = orc.q8_1_fields(orc.q8_1_quantize(x2), 3, 256)
    changed = (d != d2) | (s != s2) | (q != q2).any(axis=-1)
    assert list(zip(*np.nonzero(changed))) == [(1, 1)]
    # dequantised error is within half a step: |x - d*q| <= d/2
    deq = orc.q8_1_dequantize(q8, 3, 256).reshape(3, 8, 32)
    err = np.abs(x.reshape(3, 8, 32) - deq)
    assert np.all(err <= d[..., None].astype(np.float64) * (0.5 + 1e-6))


def test_q8_1_quotient_is_ieee_division(orc):
    """q = round(x / d) with the IEEE-754 f32 quotient (numpy's division), ties away
    from zero -- not x * (1/d), which rounds differently next to the .5 boundaries."""
    g = np.random.default_rng(9)
    nblk = 4000
    amax = g.uniform(0.01, 100, nblk).astype(np.float32)
    d = amax / np.float32(127)
    k = g.integers(-126, 126, (nblk, 31)).astype(np.float32)
    # put every element next to a rounding boundary: (k + 0.5) * d, nudged by an ulp
    x = ((k + np.float32(0.5)) * d[:, None]).astype(np.float32)
    nudge = g.integers(-1, 2, x.shape)
    x = np.where(nudge > 0, np.nextafter(x, np.float32(np.inf)),
                 np.where(nudge < 0, np.nextafter(x, np.float32(-np.inf)), x))
    x = np.concatenate([amax[:, None], x], axis=1).astype(np.float32)   # amax first
    _, _, q = orc.q8_1_fields(orc.q8_1_quantize(x.reshape(1, -1)), 1, x.size)
    q = q.reshape(nblk, 32).astype(np.float64)
    quot = (x / d[:, None]).astype(np.float64)               # f32 IEEE quotient
    expect = np.where(quot >= 0, np.floor(quot + 0.5), np.ceil(quot - 0.5))
    assert np.array_equal(q, np.clip(expect, -127, 127))
    recip = (x * (np.float32(1) / d[:, None])).astype(np.float64)
    alt = np.where(recip >= 0, np.floor(recip + 0.5), np.ceil(recip - 0.5))
    assert np.count_nonzero(alt != expect) > 10   # the two readings are distinguishable here
