"""Pins of the CPU oracle against things other than itself.

Hand-worked values (tests/golden/), closed forms, invariants of the layout,
brute force on tiny inputs, library routines (libm exp, numpy stable sort,
scipy softmax, numpy fp64 matmul) and special cases that reduce to a plain
SwiGLU MLP or a dense softmax mixture. No GPU is used.
"""
import math

import numpy as np
from scipy.special import erf
import pytest
from scipy.special import softmax

import oracle
import synth
from conftest import read_golden


def _bf16(a):
    return synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- capacity
def test_capacity_worked_values():
    rows = read_golden("capacity.txt")
    assert len(rows) >= 8
    for r in rows:
        N, K, E, cn, cd, want = (int(v) for v in r.split())
        assert oracle.capacity(N, K, E, cn, cd) == want, r


# ---------------------------------------------------------------- exp
def test_exp_within_3ulp_of_libm():
    v = np.concatenate([np.linspace(-87.0, 0.0, 400001, dtype=np.float32),
                        -np.logspace(-30, 1.9, 20001).astype(np.float32),
                        np.array([0.0, -0.0, -1e-38, -86.99, -0.5, -1.0, -2.0], np.float32)])
    got = oracle.exp_f32(v)
    ref = np.exp(v.astype(np.float64)).astype(np.float32)
    ulp = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulp.max() <= 3
    assert oracle.exp_f32(np.array([0.0], np.float32))[0] == 1.0
    assert oracle.exp_f32(np.array([-88.0, -100.0, -1e30], np.float32)).tolist() == [0.0, 0.0, 0.0]


# ---------------------------------------------------------------- router
def _router_case(E, K, logits):
    x = _bf16(np.ones((1, 1)))
    wr = np.zeros((1, E), np.float32)
    return oracle.router(x, wr, np.asarray(logits, np.float32), K, renorm=True)


def test_router_hand_worked_cases():
    for r in read_golden("router_special.txt"):
        head, lg, ids, ps = (s.split() for s in r.split("|"))
        E, K = int(head[1]), int(head[2])
        got_ids, got_p, _, _ = _router_case(E, K, [float(v) for v in lg])
        assert got_ids[0].tolist() == [int(v) for v in ids], r
        assert got_p[0].tolist() == [float(v) for v in ps], r


@pytest.mark.parametrize("N,H,E,K,use_bias", [(37, 64, 8, 2, False), (50, 128, 16, 4, True),
                                              (19, 64, 5, 5, True)])
def test_router_matches_fp64_library_routines(N, H, E, K, use_bias):
    rng = np.random.default_rng(N * 1000 + E)
    x = _bf16(rng.standard_normal((N, H)))
    wr = (rng.standard_normal((H, E)) * 0.05).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.5).astype(np.float32) if use_bias else None
    ids, p, probs, logits = oracle.router(x, wr, bias, K, renorm=True, want_probs=True,
                                          want_logits=True)
    ref_l = _f(x) @ wr.astype(np.float64) + (0 if bias is None else bias.astype(np.float64))
    assert np.allclose(logits, ref_l, rtol=0, atol=1e-4)
    ref_p = softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(probs, ref_p, rtol=1e-5, atol=1e-7)
    # top-K = first K of a stable sort on descending p (ties keep the lower e)
    order = np.argsort(-probs.astype(np.float64), axis=1, kind="stable")[:, :K]
    assert np.array_equal(ids, order)
    # renormalisation over the picks
    chosen = np.take_along_axis(probs.astype(np.float64), ids.astype(np.int64), axis=1)
    assert np.allclose(p, chosen / chosen.sum(1, keepdims=True), rtol=1e-6, atol=0)
    assert np.all(p[:, :-1] >= p[:, 1:])


# Exact fp32 arithmetic: each operation is the exact rational result rounded
# once to the nearest fp32 value, ties to the even significand (IEEE 754
# round-to-nearest-even; normal and subnormal range, no overflow here).
def _rn32(q):
    from fractions import Fraction
    if q == 0:
        return np.float32(0.0)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    scaled = a / quantum
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    v = float(m * quantum)
    return np.float32(v if q > 0 else -v)


def _q(v):
    from fractions import Fraction
    return Fraction(float(v))


def _exact_router(x, wr, bias, K, *, fused=True, ascending=True):
    """The router step by step in exact fp32 arithmetic: each logit the
    sequential chain l = fma(x[h], W_r[h,e], l) over ascending h, then + b[e];
    z = exp(l - max) with the oracle's exp (pinned to libm above); the
    denominator summed in ascending e; p = z / sum; K picks of the largest p
    (the lower e on ties); p' = p / (the picked p summed in pick order).
    fused=False / ascending=False give the plausible wrong forms the pin must
    tell apart (a rounded product before each add; descending h)."""
    xf = _f(x)
    N, H = xf.shape
    E = wr.shape[1]
    logits = np.empty((N, E), np.float32)
    probs = np.empty((N, E), np.float32)
    ids = np.empty((N, K), np.int32)
    pk = np.empty((N, K), np.float32)
    hs = range(H) if ascending else range(H - 1, -1, -1)
    for t in range(N):
        for e in range(E):
            acc = np.float32(0.0)
            for h in hs:
                if fused:
                    acc = _rn32(_q(xf[t, h]) * _q(wr[h, e]) + _q(acc))
                else:
                    acc = _rn32(_q(_rn32(_q(xf[t, h]) * _q(wr[h, e]))) + _q(acc))
            logits[t, e] = _rn32(_q(acc) + _q(0.0 if bias is None else bias[e]))
        m = max(logits[t])
        z = [oracle.exp_f32(np.array([_rn32(_q(logits[t, e]) - _q(m))], np.float32))[0]
             for e in range(E)]
        s = np.float32(0.0)
        for e in range(E):
            s = _rn32(_q(s) + _q(z[e]))
        for e in range(E):
            probs[t, e] = _rn32(_q(z[e]) / _q(s))
        taken, d = set(), np.float32(0.0)
        for k in range(K):
            best = max((e for e in range(E) if e not in taken), key=lambda e: (probs[t, e], -e))
            taken.add(best)
            ids[t, k] = best
            d = _rn32(_q(d) + _q(probs[t, best]))
        for k in range(K):
            pk[t, k] = _rn32(_q(probs[t, ids[t, k]]) / _q(d))
    return ids, pk, probs, logits


def test_router_is_the_exact_fp32_chain():
    """Bit for bit against the step-by-step definition in exact arithmetic:
    logits, softmax probabilities, picks and renormalised p'. The wrong
    forms of the logit chain (unfused, descending h) give other bits on
    these inputs, so the pin tells them apart."""
    rng = np.random.default_rng(11)
    N, H, E, K = 6, 24, 7, 3
    x = _bf16(rng.standard_normal((N, H)))
    wr = (rng.standard_normal((H, E)) * rng.choice([0.003, 0.05, 0.7], size=(H, E))).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32)
    ids, p, probs, logits = oracle.router(x, wr, bias, K, renorm=True, want_probs=True,
                                          want_logits=True)
    r_ids, r_p, r_probs, r_logits = _exact_router(x, wr, bias, K)
    assert np.array_equal(logits.view(np.uint32), r_logits.view(np.uint32))
    assert np.array_equal(probs.view(np.uint32), r_probs.view(np.uint32))
    assert np.array_equal(ids, r_ids)
    assert np.array_equal(p.view(np.uint32), r_p.view(np.uint32))
    for wrong in ({"fused": False}, {"ascending": False}):
        w_logits = _exact_router(x, wr, bias, K, **wrong)[3]
        assert not np.array_equal(w_logits.view(np.uint32), r_logits.view(np.uint32)), wrong


def _exact_exp_steps(v):
    """exp(v) by the stated method, each fp32 operation exact then rounded
    once: n = rint(v·log2 e); r = v − n·ln2_hi − n·ln2_lo (two fused steps);
    the degree-7 Taylor polynomial of e^r in Horner form (fused steps,
    coefficients 1/k! rounded from double); times 2^n. The constants follow
    their definitions: log2 e and ln 2 rounded from double to fp32, ln2_lo the
    double remainder ln 2 − ln2_hi rounded to fp32."""
    import math
    from fractions import Fraction
    if v < -87.0:
        return np.float32(0.0)
    f32 = lambda d: _rn32(Fraction(d))
    log2e, ln2_hi = f32(1.0 / math.log(2.0)), f32(math.log(2.0))
    ln2_lo = f32(math.log(2.0) - float(ln2_hi))
    y = _rn32(_q(v) * _q(log2e))
    fl = math.floor(float(y))
    n = fl + 1 if (float(y) - fl > 0.5 or (float(y) - fl == 0.5 and fl % 2 == 1)) else fl
    r = _rn32(-n * _q(ln2_hi) + _q(v))
    r = _rn32(-n * _q(ln2_lo) + _q(r))
    p = f32(1.0 / 5040.0)
    for c in (1.0 / 720.0, 1.0 / 120.0, 1.0 / 24.0, 1.0 / 6.0, 0.5, 1.0, 1.0):
        p = _rn32(_q(p) * _q(r) + _q(f32(c)))
    return _rn32(_q(p) * Fraction(2) ** n)


def test_exp_is_the_stated_method_step_by_step():
    """Bit for bit against the method evaluated in exact arithmetic (a
    coefficient or a reduction term off by a fraction of an ulp passes the
    libm bound above but not this)."""
    rng = np.random.default_rng(5)
    v = np.concatenate([-rng.uniform(0.0, 87.0, 1500), -rng.exponential(1.0, 500),
                        [0.0, -0.5, -1.0, -0.34657359, -0.34657362, -86.99, -87.0, -88.0]])
    v = v.astype(np.float32)
    got = oracle.exp_f32(v)
    want = np.array([_exact_exp_steps(float(a)) for a in v], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_router_without_renorm_returns_softmax_probs():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((20, 64)))
    wr = (rng.standard_normal((64, 8)) * 0.1).astype(np.float32)
    ids, p, probs, _ = oracle.router(x, wr, None, 3, renorm=False, want_probs=True)
    assert np.array_equal(p, np.take_along_axis(probs, ids.astype(np.int64), axis=1))


def test_router_thread_count_invariant():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_host_inputs(w, experts=[])
    n0 = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        a = oracle.router(inp["x"], inp["wr"], None, 2)
        oracle.set_num_threads(max(2, n0))
        b = oracle.router(inp["x"], inp["wr"], None, 2)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.int32), b[1].view(np.int32))


# ---------------------------------------------------------------- selection + layout
def _golden_layout(name):
    d = {}
    for r in read_golden(name):
        k, *v = r.split()
        d[k] = v
    return d


@pytest.mark.parametrize("name", ["layout_ties_k1.txt", "layout_prob_k2.txt",
                                  "layout_one_expert.txt"])
def test_layout_hand_worked(name):
    g = _golden_layout(name)
    N, E, K, cap, bm = (int(g[k][0]) for k in ("N", "E", "K", "cap", "bm"))
    ids = np.array(g["topk_ids"], np.int32).reshape(N, K)
    p = np.array(g["topk_p"], np.float32).reshape(N, K)
    L = oracle.select_layout(ids, p, E, cap, bm)
    ints = lambda k: [int(v) for v in g[k]]
    assert L.keep.ravel().tolist() == ints("keep")
    assert L.expert_counts.tolist() == ints("expert_counts")
    assert L.kept_counts.tolist() == ints("kept_counts")
    assert L.sorted_slot_ids.tolist() == ints("sorted_slot_ids")
    assert L.expert_ids.tolist() == ints("expert_ids")
    assert L.block_start.tolist() == ints("block_start")
    assert L.num_tokens_post_padded == int(g["num_tokens_post_padded"][0])
    assert L.token_routes.ravel().tolist() == ints("token_routes")


def _random_routes(rng, N, E, K, levels):
    """topk ids (distinct per token) and probabilities drawn from a few levels (many ties)."""
    ids = np.stack([rng.permutation(E)[:K] for _ in range(N)]).astype(np.int32)
    p = rng.integers(1, levels + 1, size=(N, K)).astype(np.float32) / np.float32(levels)
    return ids, p


def _brute_keep(ids, p, E, cap):
    """Route i of expert e is kept iff fewer than cap routes of e beat it on
    (p descending, token ascending): O(R^2) rank counting."""
    N, K = ids.shape
    keep = np.zeros((N, K), np.uint8)
    for t in range(N):
        for k in range(K):
            e = ids[t, k]
            better = 0
            for t2 in range(N):
                for k2 in range(K):
                    if ids[t2, k2] != e or (t2 == t and k2 == k):
                        continue
                    if p[t2, k2] > p[t, k] or (p[t2, k2] == p[t, k] and t2 < t):
                        better += 1
            keep[t, k] = better < cap
    return keep


@pytest.mark.parametrize("seed", range(6))
def test_selection_matches_brute_force_rank(seed):
    rng = np.random.default_rng(seed)
    N, E, K = int(rng.integers(1, 40)), int(rng.integers(1, 7)), 0
    K = int(rng.integers(1, E + 1))
    cap = int(rng.integers(0, N + 2))
    ids, p = _random_routes(rng, N, E, K, levels=int(rng.integers(1, 5)))
    L = oracle.select_layout(ids, p, E, cap, 16)
    assert np.array_equal(L.keep, _brute_keep(ids, p, E, cap))


def check_layout_invariants(L, ids, p, N, E, K, cap, bm):
    """Invariants of the drop-and-pad layout; returns nothing, asserts all."""
    cpad = -(-cap // bm) * bm
    assert L.cpad == cpad
    assert L.num_tokens_post_padded == E * cpad
    assert len(L.sorted_slot_ids) == E * cpad  # every expert owns exactly cpad slots
    counts = np.bincount(ids.ravel(), minlength=E)
    assert np.array_equal(L.expert_counts, counts)
    assert np.array_equal(L.kept_counts, np.minimum(counts, cap))
    assert L.keep.sum() == L.kept_counts.sum() <= min(N * K, E * cap)
    assert np.array_equal(L.block_start, np.arange(E) * cpad // bm)
    for e in range(E):
        reg = L.sorted_slot_ids[e * cpad:(e + 1) * cpad]
        kept = reg[:L.kept_counts[e]]
        assert np.all(np.diff(kept) > 0)                  # ascending token order
        assert np.all(reg[L.kept_counts[e]:] == N)        # padding holds the sentinel
        mine = (ids == e)
        assert set(kept.tolist()) == set(np.nonzero((mine & (L.keep == 1)).any(1))[0].tolist())
        pk = p[mine & (L.keep == 1)]
        pd = p[mine & (L.keep == 0)]
        if len(pk) and len(pd):
            assert pk.min() >= pd.max()                   # kept never lose to a drop
        for b in range(cpad // bm):
            blk = e * cpad // bm + b
            want = e if b * bm < L.kept_counts[e] else -1
            assert L.expert_ids[blk] == want
    # token_routes is the inverse map of the kept routes
    for t in range(N):
        for k in range(K):
            s = L.token_routes[t, k]
            if L.keep[t, k]:
                assert L.sorted_slot_ids[s] == t and s // cpad == ids[t, k]
            else:
                assert s == -1
    kept_slots = L.token_routes[L.keep == 1]
    assert len(np.unique(kept_slots)) == len(kept_slots)


@pytest.mark.parametrize("bm", [16, 32, 64, 128])
@pytest.mark.parametrize("seed", range(3))
def test_layout_invariants_random(bm, seed):
    rng = np.random.default_rng(100 + seed)
    N, E = int(rng.integers(1, 300)), int(rng.integers(1, 20))
    K = int(rng.integers(1, min(E, 6) + 1))
    cap = oracle.capacity(N, K, E, int(rng.integers(1, 5)), int(rng.integers(1, 5)))
    ids, p = _random_routes(rng, N, E, K, levels=7)
    L = oracle.select_layout(ids, p, E, cap, bm)
    check_layout_invariants(L, ids, p, N, E, K, cap, bm)


def test_layout_on_tiny_workload_invariants():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_host_inputs(w, experts=[])
    R = oracle.route(inp["x"], inp["wr"], inp["bias"], w.n_experts, w.top_k, w.cap_num,
                     w.cap_den, 32)
    check_layout_invariants(R.layout, R.topk_ids, R.topk_p, w.n_tokens, w.n_experts, w.top_k,
                            R.layout.cap, 32)
    assert R.layout.cap == 64


def test_no_drops_when_capacity_covers_all_tokens():
    rng = np.random.default_rng(7)
    N, E, K = 64, 6, 3
    ids, p = _random_routes(rng, N, E, K, levels=3)
    L = oracle.select_layout(ids, p, E, N, 16)
    assert L.keep.all() and np.array_equal(L.kept_counts, L.expert_counts)


# ---------------------------------------------------------------- FFN + combine
def _tiny_problem(rng, N, H, E, K, I, cap_num, cap_den, bm=16, wscale=0.1, act=0,
                  prob_in_act=False):
    x = _bf16(rng.standard_normal((N, H)))
    wr = (rng.standard_normal((H, E)) * 0.1).astype(np.float32)
    wg = {e: _bf16(rng.standard_normal((H, I)) * wscale) for e in range(E)}
    wu = {e: _bf16(rng.standard_normal((H, I)) * wscale) for e in range(E)}
    wd = {e: _bf16(rng.standard_normal((I, H)) * wscale) for e in range(E)}
    R = oracle.route(x, wr, None, E, K, cap_num, cap_den, bm)
    W = oracle.ExpertWeights(E, wg, wu, wd)
    y = oracle.forward_tokens(0, N, x, W, H, I, R.topk_ids, R.topk_p, R.layout.keep, act=act,
                              prob_in_act=prob_in_act)
    return x, wr, wg, wu, wd, R, y


def _swiglu_fp64(xr, wg, wu, wd, act=0):
    g = xr @ _f(wg)
    u = xr @ _f(wu)
    if act == 1:  # GELU, v * Phi(v)
        a = 0.5 * g * (1.0 + erf(g / np.sqrt(2.0))) * u
    else:
        a = g / (1.0 + np.exp(-g)) * u
    return a @ _f(wd)


@pytest.mark.parametrize("seed,act,prob_in_act", [(0, 0, False), (1, 0, False), (2, 0, False),
                                                  (3, 1, False), (4, 0, True), (5, 1, True)])
def test_forward_matches_dense_fp64_reference(seed, act, prob_in_act):
    """Every expert on every token in fp64, masked by the kept set and weighted
    by the renormalised probability, summed: equals the oracle's y (SwiGLU or
    GeGLU; the probability applied in the combine or in the activation)."""
    rng = np.random.default_rng(seed)
    N, H, E, K, I = 48, 32, 6, 2, 24
    x, wr, wg, wu, wd, R, y = _tiny_problem(rng, N, H, E, K, I, 3, 4, act=act,
                                            prob_in_act=prob_in_act)
    assert (R.layout.keep == 0).any()  # capacity factor 0.75 forces drops
    xd = _f(x)
    dense = np.stack([_swiglu_fp64(xd, wg[e], wu[e], wd[e], act) for e in range(E)])  # [E,N,H]
    ref = np.zeros((N, H))
    for t in range(N):
        for k in range(K):
            if R.layout.keep[t, k]:
                ref[t] += R.topk_p[t, k] * dense[R.topk_ids[t, k], t]
    assert np.abs(y - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
    dropped_all = ~R.layout.keep.any(1)
    assert np.all(y[dropped_all] == 0.0)


def test_single_expert_top1_is_plain_swiglu_mlp():
    rng = np.random.default_rng(11)
    N, H, I = 40, 64, 48
    x, wr, wg, wu, wd, R, y = _tiny_problem(rng, N, H, 1, 1, I, 1, 1)
    assert R.layout.keep.all() and np.all(R.topk_p == 1.0)
    ref = _swiglu_fp64(_f(x), wg[0], wu[0], wd[0])
    assert np.abs(y - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())


def test_top_k_equal_to_experts_is_dense_softmax_mixture():
    rng = np.random.default_rng(12)
    N, H, E, I = 30, 32, 4, 16
    x, wr, wg, wu, wd, R, y = _tiny_problem(rng, N, H, E, E, I, 1, 1)
    assert R.layout.keep.all()
    xd = _f(x)
    prob = softmax(xd @ wr.astype(np.float64), axis=1)
    ref = sum(prob[:, e:e + 1] * _swiglu_fp64(xd, wg[e], wu[e], wd[e]) for e in range(E))
    assert np.abs(y - ref).max() <= 2e-5 * max(1.0, np.abs(ref).max())


def test_ffn_routes_activation_output():
    rng = np.random.default_rng(5)
    H, I = 32, 16
    x = _bf16(rng.standard_normal((3, H)))
    wg, wu, wd = (_bf16(rng.standard_normal(s) * 0.2) for s in ((H, I), (H, I), (I, H)))
    W = oracle.ExpertWeights(1, {0: wg}, {0: wu}, {0: wd})
    o, h = oracle.ffn_routes([2, 0], [0, 0], x, W, H, I, want_h=True)
    xd = _f(x)[[2, 0]]
    g, u = xd @ _f(wg), xd @ _f(wu)
    a = g / (1 + np.exp(-g)) * u
    assert np.allclose(h, a, atol=1e-6) and np.allclose(o, a @ _f(wd), atol=1e-6)


def test_gelu_closed_form_values():
    """GeGLU activation a = gelu(g) * u with g = v (x = 1, one hidden unit) and
    u = 1: equals v * Phi(v) with Phi the standard normal distribution
    function, at values from its table."""
    phi = {0.0: 0.5, 0.5: 0.6914624612740131, 1.0: 0.8413447460685429, 2.0: 0.9772498680518208,
           3.0: 0.9986501019683699, -1.0: 0.15865525393145707, -2.0: 0.022750131948179195}
    vs = np.array(sorted(phi), dtype=np.float32)
    I = len(vs)
    x = _bf16(np.ones((1, 1)))
    wg = _bf16(vs[None, :])
    wu = _bf16(np.ones((1, I)))
    wd = _bf16(np.ones((I, 1)))
    W = oracle.ExpertWeights(1, {0: wg}, {0: wu}, {0: wd})
    _, h = oracle.ffn_routes([0], [0], x, W, 1, I, want_h=True, act=oracle.ACT_GELU)
    want = np.array([v * phi[float(v)] for v in vs])
    assert np.all(np.abs(h[0] - want) <= 2e-6 * np.maximum(1.0, np.abs(want)))
    # the SiLU path at the same points: v * sigma(v), sigma(0) = 1/2, and the tails
    _, hs = oracle.ffn_routes([0], [0], x, W, 1, I, want_h=True, act=oracle.ACT_SILU)
    assert hs[0][list(vs).index(0.0)] == 0.0
    assert abs(hs[0][list(vs).index(3.0)] - 3.0 / (1.0 + np.exp(-3.0))) <= 2e-6 * 3


def test_probability_in_activation_equals_in_combine():
    """p' applied to the activation (unit-weight combine) equals p' applied in
    the combine, up to fp32 rounding: the two placements of the routing weight
    ("Permute-Free Grouped GEMM for MoE (bf16, gfx950)", section 3 act*up*prob,
    or the combine) are the same function."""
    rng = np.random.default_rng(21)
    N, H, E, K, I = 40, 32, 5, 2, 16
    _, _, _, _, _, _, y0 = _tiny_problem(rng, N, H, E, K, I, 1, 1)
    rng = np.random.default_rng(21)
    _, _, _, _, _, _, y1 = _tiny_problem(rng, N, H, E, K, I, 1, 1, prob_in_act=True)
    assert np.abs(y0 - y1).max() <= 1e-6 * max(1.0, np.abs(y0).max())
