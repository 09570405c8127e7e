"""Pins of the oracle's FP8 path (E4M3: 1 sign, 4 exponent bits with bias 7,
3 mantissa bits, max 448, no infinities): decoded values from the format's
definition, encoding by round-to-nearest-even with saturation, row-wise
quantisation, and FC1 on the quantised operands against fp64. No GPU."""
import numpy as np
import pytest

import oracle
import synth


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x30, 0.5), (0x3C, 1.5), (0x40, 2.0), (0xC0, -2.0), (0x7E, 448.0),
    (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x39, 1.125), (0x77, 240.0),
])
def test_e4m3_decode_table(code, value):
    assert oracle.e4m3_decode([code])[0] == np.float32(value)


def test_e4m3_nan_and_round_trip():
    assert np.isnan(oracle.e4m3_decode([0x7F])[0]) and np.isnan(oracle.e4m3_decode([0xFF])[0])
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)
    # decoded values increase with the code on the positive side
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


@pytest.mark.parametrize("value,code", [
    (1.0625, 0x38),            # midpoint of 1 and 1.125: to the even code
    (1.1875, 0x3A),            # midpoint of 1.125 and 1.25: to the even code
    (1.07, 0x39), (1.05, 0x38),
    (500.0, 0x7E), (-1e9, 0xFE), (448.0, 0x7E), (460.0, 0x7E),   # saturation
    (2.0 ** -10, 0x00),        # half the smallest subnormal: tie, to the even code 0
    (0.75 * 2.0 ** -9, 0x01), (3 * 2.0 ** -10, 0x02),            # 1.5 x 2^-9: tie between 1 and 2
    (-0.3, 0xAA),              # -0.3 lies between -0.28125 (0xA9) and -0.3125 (0xAA): 0.0125
                               # from the second, 0.01875 from the first
])
def test_e4m3_encode_rounding(value, code):
    assert oracle.e4m3_encode([value])[0] == code


def test_e4m3_encode_is_nearest_code_for_every_bf16_value():
    """Every bf16 value of magnitude up to 450, both signs: the code is the
    nearest finite value by exhaustive search over the decoded table, ties to
    the even code, saturation at 448."""
    vals = synth.bf16_bits_to_f32(np.arange(0, 0x43E1, dtype=np.uint16)).astype(np.float64)
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    d = np.abs(table[None, :] - np.minimum(vals, 448.0)[:, None])
    best = d.min(axis=1, keepdims=True)
    ties = d == best
    # the lowest even candidate when two tie, else the only one
    even = ties & (np.arange(0x7F)[None, :] % 2 == 0)
    expect = np.where(ties.sum(axis=1) > 1, even.argmax(axis=1), ties.argmax(axis=1)).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(vals), expect)
    assert np.array_equal(oracle.e4m3_encode(-vals[1:]), expect[1:] | 0x80)


def test_quantize_rows_scale_and_extremes():
    rng = np.random.default_rng(0)
    m = synth.f32_to_bf16_bits(rng.standard_normal((6, 40)).astype(np.float32) * 3)
    m[2] = 0  # an all-zero row
    q, s = oracle.quantize_rows_fp8(m)
    f = synth.bf16_bits_to_f32(m)
    for r in range(6):
        amax = np.abs(f[r]).max()
        if amax == 0:
            assert s[r] == 1.0 and np.all(q[r] == 0)
            continue
        assert s[r] == np.float32(amax) / np.float32(448.0)
        # the largest magnitude quantises to +-448
        assert oracle.e4m3_decode([q[r][np.abs(f[r]).argmax()]])[0] in (448.0, -448.0)
        # quantisation error within half an E4M3 step (relative 2^-4) of the scaled value
        deq = oracle.e4m3_decode(q[r]).astype(np.float64) * s[r]
        assert np.all(np.abs(deq - f[r]) <= 2.0 ** -4 * np.abs(f[r]) + 2.0 ** -10 * s[r])


@pytest.mark.parametrize("act", [0, 1])
def test_fc1_fp8_matches_fp64_dequantised_reference(act):
    from scipy.special import erf
    rng = np.random.default_rng(3 + act)
    N, H, E, I = 7, 64, 3, 32
    x = synth.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    w13 = synth.f32_to_bf16_bits((rng.standard_normal((E * 2 * I, H)) * 0.1).astype(np.float32))
    xq, xs = oracle.quantize_rows_fp8(x)
    wq, ws = oracle.quantize_rows_fp8(w13)
    toks = np.array([0, 3, 6, 2], np.int32)
    exps = np.array([1, 0, 2, 1], np.int32)
    h = oracle.fc1_fp8_routes(toks, exps, xq, xs, wq.reshape(E, 2 * I, H), ws.reshape(E, 2 * I), H, I,
                              act=act)
    X = oracle.e4m3_decode(xq).astype(np.float64) * xs[:, None]
    W = oracle.e4m3_decode(wq).astype(np.float64) * ws[:, None]
    for j, (t, e) in enumerate(zip(toks, exps)):
        g = W[e * 2 * I:e * 2 * I + I] @ X[t]
        u = W[e * 2 * I + I:(e + 1) * 2 * I] @ X[t]
        a = 0.5 * g * (1 + erf(g / np.sqrt(2))) if act == 1 else g / (1 + np.exp(-g))
        ref = a * u
        assert np.abs(h[j] - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())


def test_fc2_fp8_matches_fp64_dequantised_reference():
    rng = np.random.default_rng(11)
    n, H, E, I = 5, 48, 3, 64
    h = synth.f32_to_bf16_bits(rng.standard_normal((n, I)).astype(np.float32))
    w2 = synth.f32_to_bf16_bits((rng.standard_normal((E * H, I)) * 0.1).astype(np.float32))
    hq, hs = oracle.quantize_rows_fp8(h)
    wq, ws = oracle.quantize_rows_fp8(w2)
    exps = np.array([2, 0, 1, 2, 0], np.int32)
    o = oracle.fc2_fp8_routes(exps, hq, hs, wq.reshape(E, H, I), ws.reshape(E, H), H, I)
    Hd = oracle.e4m3_decode(hq).astype(np.float64) * hs[:, None]
    W = oracle.e4m3_decode(wq).astype(np.float64) * ws[:, None]
    for j, e in enumerate(exps):
        ref = W[e * H:(e + 1) * H] @ Hd[j]
        assert np.abs(o[j] - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
    # dequantised operands stay within the quantisation error of the bf16 product
    full = synth.bf16_bits_to_f32(w2).astype(np.float64).reshape(E, H, I)
    hf = synth.bf16_bits_to_f32(h).astype(np.float64)
    for j, e in enumerate(exps):
        exact = full[e] @ hf[j]
        assert np.abs(o[j] - exact).max() <= 0.15 * np.abs(exact).max()
