"""Pins of the oracle's MX block-scaled FP8 path (MXFP8 E4M3 as the OCP
Microscaling Formats v1.0 specification defines it; no page defines a
block-scaled format): E8M0 scale codes from the definition, the block scale
exponent floor(log2 amax) - 8 on worked values, element codes against an
exhaustive nearest-value search done here in float64, the error bound of one
block, independence of the blocks, and FC1 / FC2 on MX operands against fp64
products of the dequantised operands. No GPU."""
import numpy as np
import pytest

import oracle
import synth

E4M3_TABLE = None


def e4m3_table():
    """Non-negative finite E4M3 values by code (0x00..0x7E), from the format's
    definition: subnormal m/8 * 2^-6, normal (1 + m/8) * 2^(e-7)."""
    global E4M3_TABLE
    if E4M3_TABLE is None:
        v = []
        for c in range(0x7F):
            e, m = c >> 3, c & 7
            v.append(m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
        E4M3_TABLE = np.array(v)
    return E4M3_TABLE


def nearest_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest code by search over the table, ties to the even code, |x| >= 448
    saturates, the sign bit kept (a negative value that rounds to zero gives
    0x80); x in float64."""
    t = e4m3_table()
    a = np.minimum(np.abs(x), 448.0)
    d = np.abs(t[None, :] - a[:, None])
    best = d.min(axis=1, keepdims=True)
    ties = d == best
    even = ties & (np.arange(0x7F)[None, :] % 2 == 0)
    code = np.where(ties.sum(axis=1) > 1, even.argmax(axis=1), ties.argmax(axis=1)).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def bf16(values) -> np.ndarray:
    return synth.f32_to_bf16_bits(np.asarray(values, np.float32))


@pytest.mark.parametrize("code,value", [(127, 1.0), (128, 2.0), (126, 0.5), (0, 2.0 ** -127),
                                        (254, 2.0 ** 127), (100, 2.0 ** -27), (119, 2.0 ** -8)])
def test_e8m0_decode(code, value):
    assert oracle.e8m0_decode([code])[0] == np.float32(value)


def test_e8m0_nan():
    assert np.isnan(oracle.e8m0_decode([255])[0])


@pytest.mark.parametrize("amax,code", [
    (1.0, 119),            # floor(log2 1) - 8 = -8
    (448.0, 127),          # floor(log2 448) = 8 -> 2^0
    (0.75, 118),           # floor(log2 0.75) = -1 -> 2^-9
    (1.9921875, 119),      # just below 2: still exponent 0
    (2.0, 120),
    (1e30, 127 + 99 - 8),  # bf16(1e30) = 1.0005... * 2^99
    (2.0 ** -130, 0),      # -138 clamped to -127
])
def test_block_scale_exponent_worked_values(amax, code):
    row = np.zeros(32, np.float32)
    row[5] = amax
    row[9] = -amax / 3
    q, sc = oracle.quantize_mx_fp8(bf16(row)[None, :])
    assert sc[0, 0] == code


def test_all_zero_block_and_saturation():
    q, sc = oracle.quantize_mx_fp8(bf16(np.zeros((1, 64))))
    assert np.all(sc == 0) and np.all(q == 0)
    # a block maximum of 500 = 1.95 * 2^8: scale 2^0, the maximum saturates to 448
    row = np.linspace(-3, 3, 32).astype(np.float32)
    row[7] = 500.0
    q, sc = oracle.quantize_mx_fp8(bf16(row)[None, :])
    assert sc[0, 0] == 127 and q[0, 7] == 0x7E
    row[7] = -500.0
    q, _ = oracle.quantize_mx_fp8(bf16(row)[None, :])
    assert q[0, 7] == 0xFE


def test_codes_are_nearest_e4m3_of_the_scaled_values():
    """Random rows with a spread of magnitudes per block: every code is the
    nearest E4M3 value of v / 2^s found by exhaustive search in float64, with
    s taken from the stored scale code."""
    rng = np.random.default_rng(3)
    rows, cols = 40, 256
    mag = np.exp2(rng.integers(-20, 20, size=(rows, cols // 32)).astype(np.float64))
    v = rng.standard_normal((rows, cols)) * np.repeat(mag, 32, axis=1)
    v[0, :32] = 0.0                       # an all-zero block
    v[1, 32:64] = [(-1) ** i * 2.0 ** (i - 16) for i in range(32)]  # exact powers of two
    bits = bf16(v.astype(np.float32))
    vb = synth.bf16_bits_to_f32(bits).astype(np.float64)
    q, sc = oracle.quantize_mx_fp8(bits)
    s = sc.astype(np.int64) - 127
    # the scale exponent from the block maxima, recomputed here
    amax = np.abs(vb).reshape(rows, cols // 32, 32).max(axis=2)
    want_s = np.clip(np.floor(np.log2(np.where(amax > 0, amax, 1.0))).astype(np.int64) - 8, -127, 127)
    want_s[amax == 0] = -127
    assert np.array_equal(s, want_s)
    scaled = vb / np.exp2(np.repeat(s, 32, axis=1))
    assert np.array_equal(q.ravel(), nearest_e4m3(scaled.ravel()))


def test_dequantisation_error_bound():
    """A non-saturated element is within half an E4M3 step of its value: the
    step is 2^(e-3) for a normal result of exponent e and 2^-9 for a
    subnormal one, times the block scale; a saturated one (|v| / 2^s in
    [448, 512)) is off by less than 64 * 2^s."""
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 128)) * 10.0 ** rng.uniform(-3, 3, size=(64, 1))
    bits = bf16(v.astype(np.float32))
    vb = synth.bf16_bits_to_f32(bits).astype(np.float64)
    q, sc = oracle.quantize_mx_fp8(bits)
    X = np.repeat(oracle.e8m0_decode(sc.ravel()).reshape(sc.shape).astype(np.float64), 32, axis=1)
    deq = oracle.e4m3_decode(q.ravel()).reshape(q.shape).astype(np.float64) * X
    r = np.abs(vb) / X
    sat = r > 448.0
    e = np.floor(np.log2(np.maximum(r, 2.0 ** -6)))
    half_step = np.where(r < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4)) * X
    assert np.all(np.abs(deq - vb)[~sat] <= half_step[~sat])
    assert np.all(np.abs(deq - vb)[sat] < 64.0 * X[sat])
    assert np.all(r < 512.0)


def test_blocks_are_independent():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((3, 128)).astype(np.float32)
    q0, s0 = oracle.quantize_mx_fp8(bf16(v))
    v2 = v.copy()
    v2[1, 32:64] *= 1000.0
    q1, s1 = oracle.quantize_mx_fp8(bf16(v2))
    changed = np.zeros_like(s0, bool)
    changed[1, 1] = True
    assert np.array_equal(s0[~changed], s1[~changed]) and s1[1, 1] == s0[1, 1] + 10 - \
        (0 if s0[1, 1] + 10 <= 254 else 0)
    mask = np.ones_like(q0, bool)
    mask[1, 32:64] = False
    assert np.array_equal(q0[mask], q1[mask])


def test_block_scales_beat_row_scales_on_an_outlier():
    """One large value per row: the row-wise scale flushes the rest of the row
    to a few codes, the block scales keep every other block's precision."""
    rng = np.random.default_rng(9)
    v = rng.standard_normal((16, 512)).astype(np.float32)
    v[:, 3] = 1.0e6
    bits = bf16(v)
    vb = synth.bf16_bits_to_f32(bits).astype(np.float64)
    qm, sm = oracle.quantize_mx_fp8(bits)
    Xm = np.repeat(oracle.e8m0_decode(sm.ravel()).reshape(sm.shape).astype(np.float64), 32, axis=1)
    dm = oracle.e4m3_decode(qm.ravel()).reshape(qm.shape) * Xm
    qr, sr = oracle.quantize_rows_fp8(bits)
    dr = oracle.e4m3_decode(qr.ravel()).reshape(qr.shape) * sr[:, None]
    rest = np.ones(v.shape, bool)
    rest[:, :32] = False
    err_mx = np.linalg.norm((dm - vb)[rest]) / np.linalg.norm(vb[rest])
    err_row = np.linalg.norm((dr - vb)[rest]) / np.linalg.norm(vb[rest])
    assert err_mx < 0.04 and err_row > 5 * err_mx


def _mx_operands(seed, n_tok, H, I, E):
    rng = np.random.default_rng(seed)
    x = bf16(rng.standard_normal((n_tok, H)) * np.exp2(rng.integers(-4, 4, size=(n_tok, 1))))
    wg = bf16(rng.standard_normal((E, 2 * I, H)) * 0.05)
    xq, xs = oracle.quantize_mx_fp8(x)
    wq, ws = oracle.quantize_mx_fp8(wg.reshape(E * 2 * I, H))
    return rng, xq, xs, wq.reshape(E, 2 * I, H), ws


def _deq(q, s):
    X = np.repeat(oracle.e8m0_decode(s.ravel()).reshape(s.shape).astype(np.float64), 32, axis=1)
    return oracle.e4m3_decode(q.reshape(q.shape[0], -1).ravel()).reshape(q.shape[0], -1).astype(np.float64) * X


@pytest.mark.parametrize("act", [0, 1])
def test_fc1_mx_matches_fp64_dequantised_reference(act):
    H, I, E, n_tok = 128, 64, 3, 9
    rng, xq, xs, wq, ws = _mx_operands(11 + act, n_tok, H, I, E)
    tokens = rng.integers(0, n_tok, size=12).astype(np.int32)
    experts = rng.integers(0, E, size=12).astype(np.int32)
    h = oracle.fc1_mx_routes(tokens, experts, xq, xs, wq, ws, H, I, act=act)
    xd = _deq(xq, xs)
    wd = _deq(wq.reshape(E * 2 * I, H), ws).reshape(E, 2 * I, H)
    for j, (t, e) in enumerate(zip(tokens, experts)):
        g = wd[e, :I] @ xd[t]
        u = wd[e, I:] @ xd[t]
        a = g / (1 + np.exp(-g)) if act == 0 else 0.5 * g * (1 + np.vectorize(__import__("math").erf)(g / np.sqrt(2)))
        ref = a * u
        scale = np.sqrt(np.sum((np.abs(wd[e, :I]) @ np.abs(xd[t])) ** 2) / I) + 1e-30
        assert np.max(np.abs(h[j] - ref)) <= 1e-5 * max(1.0, scale) * 10, (j, np.max(np.abs(h[j] - ref)))


def test_fc2_mx_matches_fp64_dequantised_reference():
    H, I, E, n = 96, 128, 4, 10
    rng = np.random.default_rng(21)
    hb = bf16(rng.standard_normal((n, I)) * np.exp2(rng.integers(-6, 6, size=(n, 4)).repeat(32, axis=1)))
    w2 = bf16(rng.standard_normal((E, H, I)) * 0.03)
    hq, hs = oracle.quantize_mx_fp8(hb)
    wq, ws = oracle.quantize_mx_fp8(w2.reshape(E * H, I))
    experts = rng.integers(0, E, size=n).astype(np.int32)
    o = oracle.fc2_mx_routes(experts, hq, hs, wq.reshape(E, H, I), ws, H, I)
    hd = _deq(hq, hs)
    wd = _deq(wq, ws).reshape(E, H, I)
    for j, e in enumerate(experts):
        ref = wd[e] @ hd[j]
        mag = np.abs(wd[e]) @ np.abs(hd[j])
        assert np.all(np.abs(o[j] - ref) <= 1e-6 * mag * 8 + 1e-30), j


def test_mx_layer_close_to_bf16_layer():
    """FC1 then FC2 on MX operands against the bf16 oracle on the same inputs:
    quantisation error only (a few percent relative Frobenius)."""
    w = synth.Workload("mx_close", 64, 256, 4, 2, 128, 1, 1)
    inp = synth.make_host_inputs(w)
    R = oracle.route(inp["x"], inp["wr"], None, w.n_experts, w.top_k, 1, 1, 16)
    W = oracle.ExpertWeights(w.n_experts, inp["wg"], inp["wu"], inp["wd"])
    r = np.nonzero(R.layout.token_routes.ravel() >= 0)[0]
    tok, ex = (r // w.top_k).astype(np.int32), R.topk_ids.ravel()[r].astype(np.int32)
    o_ref, h_ref = oracle.ffn_routes(tok, ex, inp["x"], W, w.hidden, w.inter, want_h=True)
    E, H, I = w.n_experts, w.hidden, w.inter
    w13 = np.concatenate([np.stack([inp["wg"][e].T for e in range(E)]),
                          np.stack([inp["wu"][e].T for e in range(E)])], axis=1)  # [E,2I,H]
    w2 = np.stack([inp["wd"][e].T for e in range(E)])                            # [E,H,I]
    xq, xs = oracle.quantize_mx_fp8(inp["x"])
    wq, ws = oracle.quantize_mx_fp8(np.ascontiguousarray(w13).reshape(E * 2 * I, H))
    h = oracle.fc1_mx_routes(tok, ex, xq, xs, wq.reshape(E, 2 * I, H), ws, H, I)
    assert np.linalg.norm(h - h_ref) / np.linalg.norm(h_ref) < 0.06
    hq, hs = oracle.quantize_mx_fp8(synth.f32_to_bf16_bits(h))
    w2q, w2s = oracle.quantize_mx_fp8(np.ascontiguousarray(w2).reshape(E * H, I))
    o = oracle.fc2_mx_routes(ex, hq, hs, w2q.reshape(E, H, I), w2s, H, I)
    assert np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref) < 0.08
