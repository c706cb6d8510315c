"""Pins of the oracle's MX FP8 quantiser (no GPU).

The quantiser follows reading R22 (OCP Microscaling FP8: E4M3 elements, one
power-of-two scale per 32 elements).  It is pinned here by the E4M3
definition itself -- every finite code round-trips, the extreme and boundary
values have their closed-form codes, rounding is to the nearest value with
ties to the even mantissa (checked against an exhaustive search over all
finite values), saturation at 448 -- by the block-scale rule (the block
maximum lands in [256, 448]), by an error bound, and by planted mistakes."""

import math

import numpy as np
import pytest

from oracle import mxfp8 as mx


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = mx.e4m3_decode(codes)
    assert np.array_equal(mx.e4m3_round(vals), vals)
    enc = mx.e4m3_encode(vals)
    # +0 and -0 are the only values with two codes; both survive
    assert np.array_equal(enc, codes)


@pytest.mark.parametrize("value,code", [
    (0.0, 0x00), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE),
    (2.0 ** -9, 0x01),            # smallest subnormal: m = 1, exponent field 0
    (7 * 2.0 ** -9, 0x07),        # largest subnormal
    (2.0 ** -6, 0x08),            # smallest normal
    (256.0, 0x78), (1.875, 0x3F), (0.5, 0x30),
])
def test_closed_form_codes(value, code):
    assert int(mx.e4m3_encode(np.array([value]))[0]) == code
    assert float(mx.e4m3_decode(np.uint8(code))) == value


def test_finite_value_set():
    v = mx.finite_values()
    assert v.size == 253            # 2 * 127 finite codes, +0 and -0 equal
    assert v.max() == 448.0 and v.min() == -448.0
    pos = v[v > 0]
    assert pos.min() == 2.0 ** -9


@pytest.mark.parametrize("v,want", [
    (1.0625, 1.0),                  # halfway 1.0 | 1.125: even mantissa (000) wins
    (1.1875, 1.25),                 # halfway 1.125 | 1.25: 1.25 (mantissa 010)
    (1.5 * 2.0 ** -9, 2 * 2.0 ** -9),   # subnormal tie -> even
    (0.5 * 2.0 ** -9, 0.0),         # half the smallest subnormal -> 0
    (7.5 * 2.0 ** -9, 2.0 ** -6),   # between largest subnormal and smallest normal
    (460.0, 448.0), (1.0e6, 448.0), (-500.0, -448.0),   # saturation
    (440.0, 448.0), (431.0, 416.0),
])
def test_rounding_ties_and_saturation(v, want):
    assert float(mx.e4m3_round(np.array([v]))[0]) == want


def test_rounding_equals_exhaustive_nearest_search():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.normal(0, 1, 400), rng.normal(0, 300, 200), rng.uniform(-2 ** -6, 2 ** -6, 200),
        mx.finite_values()[:-1] + np.diff(mx.finite_values()) / 2,   # every midpoint
    ])
    got = mx.e4m3_round(vals)
    want = np.array([mx.nearest_by_search(float(v)) for v in vals])
    assert np.array_equal(got, want)


def test_block_scale_puts_the_maximum_in_range():
    rng = np.random.default_rng(3)
    a = (rng.normal(0, 1, (64, 96)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    codes, scales = mx.quantize(a)
    assert scales.shape == (64, 3)
    s = scales.astype(np.int64) - 127
    blocks = np.abs(a.astype(np.float64)).reshape(64, 3, 32).max(axis=-1)
    scaled = blocks / np.exp2(s)
    # floor(log2 amax) - 8 as the exponent: the largest scaled element lies in [256, 512)
    assert np.all(scaled >= 256.0) and np.all(scaled < 512.0)
    assert np.all(np.abs(mx.e4m3_decode(codes)).reshape(64, 3, 32).max(axis=-1) >= 256.0)


def test_block_of_ones_and_zero_block():
    a = np.zeros((2, 64), np.float32)
    a[0, :32] = 1.0
    codes, scales = mx.quantize(a)
    assert scales[0, 0] == 127 - 8            # 2^-8: 1.0 is stored as 256 (code 0x78)
    assert np.all(codes[0, :32] == 0x78)
    assert scales[0, 1] == 0 and scales[1, 0] == 0   # all-zero blocks: s = -127
    assert np.all(codes[1] == 0)
    assert np.array_equal(mx.dequantize(codes, scales), a.astype(np.float64))


def test_dequantisation_error_bound():
    """|dq(v) - v| <= max(2^-4 |v|, 2^-10 X) inside the range (half a quantum
    of a 3-bit mantissa, or half the smallest subnormal step), and the
    saturated part of a block's top octave costs at most 64 X."""
    rng = np.random.default_rng(11)
    a = rng.normal(0, 1, (50, 256)).astype(np.float32)
    codes, scales = mx.quantize(a)
    X = np.repeat(np.exp2(scales.astype(np.float64) - 127), 32, axis=1)
    err = np.abs(mx.dequantize(codes, scales) - a.astype(np.float64))
    v = np.abs(a.astype(np.float64))
    inside = v / X <= 448.0
    assert np.all(err[inside] <= np.maximum(2.0 ** -4 * v[inside], 2.0 ** -10 * X[inside]))
    assert np.all(err[~inside] <= 64.0 * X[~inside])


def test_ragged_last_block():
    a = np.linspace(-3, 3, 70, dtype=np.float32)[None, :]
    codes, scales = mx.quantize(a)
    assert codes.shape == (1, 70) and scales.shape == (1, 3)
    # the 6-element tail block has its own maximum: |2.74| .. 3 -> s = 1 - 8
    assert scales[0, 2] == 127 - 7


# ---------------------------------------------------------------- planted mistakes
def test_truncation_instead_of_nearest_fails_the_search_pin():
    vals = np.array([1.1, 1.2, 3.3, 0.07, 250.0])
    trunc = np.copysign(np.floor(np.abs(vals) / np.exp2(np.floor(np.log2(np.abs(vals))) - 3))
                        * np.exp2(np.floor(np.log2(np.abs(vals))) - 3), vals)
    want = np.array([mx.nearest_by_search(float(v)) for v in vals])
    assert not np.array_equal(trunc, want)
    assert np.array_equal(mx.e4m3_round(vals), want)


def test_wrong_scale_exponent_fails_the_range_pin():
    """With emax 7 instead of 8 the block maximum lands in [128, 256): the
    top E4M3 octave is never used, a plausible off-by-one the range pin sees."""
    amax = np.array([1.0, 3.7, 0.02])
    _, ex = np.frexp(amax)
    wrong = amax / np.exp2(ex - 1 - 7)
    right = amax / np.exp2(mx.block_scale_exponent(amax))
    assert np.all(wrong < 256.0)
    assert np.all((right >= 256.0) & (right < 512.0))


def test_fake_quant_is_idempotent():
    rng = np.random.default_rng(5)
    a = rng.normal(0, 2, (8, 64)).astype(np.float32)
    q = mx.fake_quant(a)
    assert np.array_equal(mx.fake_quant(q.astype(np.float32)), q)
    assert math.isclose(float(np.linalg.norm(q - a) / np.linalg.norm(a)), 0.0, abs_tol=0.05)


# ---------------------------------------------------------------- the MX FP8 layer
from oracle import moe_oracle as om  # noqa: E402


def _scalar_fake_quant(row):
    """Element-by-element restatement of MX quantisation for the layer pin:
    math.frexp for the block maximum's exponent, exhaustive nearest search
    for each element."""
    out = []
    for b0 in range(0, len(row), 32):
        blk = [float(np.float32(v)) for v in row[b0:b0 + 32]]
        amax = max(abs(v) for v in blk)
        if amax == 0.0:
            s = -127
        else:
            _, e = math.frexp(amax)
            s = max(min(e - 1 - 8, 127), -127)
        X = 2.0 ** s
        out += [mx.nearest_by_search(v / X) * X for v in blk]
    return np.array(out)


def _tiny_layer(act="gelu"):
    rng = np.random.default_rng(21)
    T, d, F = 3, 64, 96
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    F1 = 2 * F if act == "swiglu" else F
    w1 = (rng.normal(0, 1, (F1, d)) / 8).astype(np.float32)
    w2 = (rng.normal(0, 1, (d, F)) / 10).astype(np.float32)
    return x, w1, w2


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_mx_expert_equals_elementwise_brute_force(act):
    x, w1, w2 = _tiny_layer(act)
    xq = np.stack([_scalar_fake_quant(r) for r in x])
    w1q = np.stack([_scalar_fake_quant(r) for r in w1])
    w2q = np.stack([_scalar_fake_quant(r) for r in w2])
    h = xq @ w1q.T
    if act == "gelu":
        h = np.array([[0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in r] for r in h])
    else:
        F = h.shape[1] // 2
        g, u = h[:, :F], h[:, F:]
        h = g / (1 + np.exp(-g)) * u
    hq = np.stack([_scalar_fake_quant(r) for r in h.astype(np.float32)])
    want = hq @ w2q.T
    got = om.expert_ffn_mxfp8(x.astype(np.float64), w1, None, w2, None, act=act)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_mx_layer_with_one_expert_is_the_mx_expert():
    """E = 1, k = 1: the layer output is the single MX expert's output (gate
    weight 1), computed through the whole oracle layer."""
    x, w1, w2 = _tiny_layer()
    cfg = om.OracleConfig(T=3, d_model=64, d_ff=96, E=1, k=1, experts="mxfp8")
    res = om.moe_forward(cfg, x.astype(np.float64), np.zeros((64, 1)),
                         lambda e: (w1.astype(np.float64), None, w2.astype(np.float64), None))
    want = om.expert_ffn_mxfp8(x.astype(np.float64), w1, None, w2, None)
    np.testing.assert_array_equal(res.out, want)


def test_mx_layer_is_close_to_the_dense_layer_but_not_equal():
    x, w1, w2 = _tiny_layer()
    dense = om.expert_ffn(x.astype(np.float64), w1, None, w2, None)
    q = om.expert_ffn_mxfp8(x.astype(np.float64), w1, None, w2, None)
    rel = np.linalg.norm(q - dense) / np.linalg.norm(dense)
    assert 1e-3 < rel < 0.1


@pytest.mark.parametrize("mistake", ["w1_wrong_axis", "h_not_quantised", "x_not_quantised"])
def test_planted_layer_mistakes_fail_the_brute_force(mistake):
    x, w1, w2 = _tiny_layer()
    x64 = x.astype(np.float64)
    xq = x64 if mistake == "x_not_quantised" else mx.fake_quant(x)
    w1q = mx.fake_quant(w1.T).T if mistake == "w1_wrong_axis" else mx.fake_quant(w1)
    h = om.gelu(xq @ w1q.T)
    hq = h if mistake == "h_not_quantised" else mx.fake_quant(h.astype(np.float32))
    wrong = hq @ mx.fake_quant(w2).T
    right = om.expert_ffn_mxfp8(x64, w1, None, w2, None)
    assert not np.allclose(wrong, right, rtol=1e-9, atol=1e-9)
