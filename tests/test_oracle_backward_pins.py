"""Pins of the oracle's dropless layout and expert-path backward.

Hand-worked layout (tests/golden/layout_dropless.txt), ladder invariants, and
central finite differences in fp64 of the forward written with numpy, for every
backward output (dX, dW_gate, dW_up, dW_down, dprob), plus an fp64 closed form
of the weight gradients on tiny inputs. No GPU."""
import numpy as np
from scipy.special import erf
import pytest

import oracle
import synth
from conftest import read_golden


def _bf16(a):
    return synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def test_dropless_layout_hand_worked():
    g = {}
    for r in read_golden("layout_dropless.txt"):
        k, *v = r.split()
        g[k] = [int(x) for x in v]
    N, E, K, bm = g["N"][0], g["E"][0], g["K"][0], g["bm"][0]
    L = oracle.dropless_layout(np.array(g["topk_ids"], np.int32).reshape(N, K), E, bm,
                               g["ladder_num"], g["ladder_den"][0])
    assert L.expert_counts.tolist() == g["expert_counts"]
    assert L.extents.tolist() == g["extents"]
    assert L.block_start.tolist() == g["block_start"]
    assert L.num_tokens_post_padded == g["num_tokens_post_padded"][0]
    assert L.sorted_slot_ids.tolist() == g["sorted_slot_ids"]
    assert L.expert_ids.tolist() == g["expert_ids"]
    assert L.token_routes.ravel().tolist() == g["token_routes"]


@pytest.mark.parametrize("seed", range(4))
def test_dropless_layout_invariants(seed):
    rng = np.random.default_rng(seed)
    N, E, K, bm = int(rng.integers(1, 200)), int(rng.integers(1, 12)), 0, int(rng.choice([16, 32, 64]))
    K = int(rng.integers(1, min(E, 4) + 1))
    # skewed routing so some experts overflow the top rung
    w = 1.0 / np.arange(1, E + 1) ** 1.2
    ids = np.stack([rng.choice(E, K, replace=False, p=w / w.sum()) for _ in range(N)]).astype(np.int32)
    ladder = [2, 3, 4, 5, 6, 8]  # 0.5x .. 2x of the expected rows, den 4
    L = oracle.dropless_layout(ids, E, bm, ladder, 4)
    R = N * K
    counts = np.bincount(ids.ravel(), minlength=E)
    assert np.array_equal(L.expert_counts, counts)
    rungs = [-(-(-(-m * R // (4 * E))) // bm) * bm for m in ladder]
    for e in range(E):
        holding = [r for r in rungs if counts[e] <= r]
        want = min(holding) if holding else -(-counts[e] // bm) * bm
        assert L.extents[e] == want
    assert np.array_equal(L.block_start * bm, np.concatenate([[0], np.cumsum(L.extents)[:-1]]))
    assert L.num_tokens_post_padded == L.extents.sum() <= len(L.sorted_slot_ids)
    for e in range(E):
        b0 = L.block_start[e] * bm
        reg = L.sorted_slot_ids[b0:b0 + L.extents[e]]
        toks = reg[:counts[e]]
        assert np.all(np.diff(toks) > 0) and np.all(reg[counts[e]:] == N)
        assert set(toks.tolist()) == set(np.nonzero((ids == e).any(1))[0].tolist())
    assert np.all(L.sorted_slot_ids[L.num_tokens_post_padded:] == N)
    assert np.all(L.token_routes >= 0)  # nothing dropped
    t = np.repeat(np.arange(N), K)
    assert np.array_equal(L.sorted_slot_ids[L.token_routes.ravel()], t)


# ---------------------------------------------------------------- backward
def _problem(seed, N=12, H=16, E=3, K=2, I=8):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((N, H)))
    dy = _bf16(rng.standard_normal((N, H)))
    wg = {e: _bf16(rng.standard_normal((H, I)) * 0.3) for e in range(E)}
    wu = {e: _bf16(rng.standard_normal((H, I)) * 0.3) for e in range(E)}
    wd = {e: _bf16(rng.standard_normal((I, H)) * 0.3) for e in range(E)}
    ids = np.stack([rng.permutation(E)[:K] for _ in range(N)]).astype(np.int32)
    p = rng.random((N, K)).astype(np.float32)
    p /= p.sum(1, keepdims=True)
    p = p.astype(np.float32)
    L = oracle.dropless_layout(ids, E, 16, [2, 4], 4)
    W = oracle.ExpertWeights(E, wg, wu, wd)
    return x, dy, wg, wu, wd, ids, p, L, W


def _loss64(x, wg, wu, wd, ids, p, dy, act=0):
    """L = sum_t <dY[t], y[t]>, y[t] = sum_k p[t,k] * FFN_{e}(x[t]) in fp64
    (act 0: SwiGLU, 1: GeGLU with the erf form of GELU)."""
    N, K = ids.shape
    y = np.zeros((N, x.shape[1]))
    for t in range(N):
        for k in range(K):
            e = ids[t, k]
            g = x[t] @ wg[e]
            u = x[t] @ wu[e]
            if act == 1:
                a = 0.5 * g * (1.0 + erf(g / np.sqrt(2.0))) * u
            else:
                a = g / (1.0 + np.exp(-g)) * u
            y[t] += p[t, k] * (a @ wd[e])
    return float((dy * y).sum())


@pytest.mark.parametrize("seed", range(2))
def test_backward_matches_central_differences(seed):
    _central_differences(seed, act=0)


@pytest.mark.parametrize("seed", range(2))
def test_backward_matches_central_differences_gelu(seed):
    _central_differences(10 + seed, act=1)


def _central_differences(seed, act):
    x, dy, wg, wu, wd, ids, p, L, W = _problem(seed)
    N, H = x.shape
    E, I = len(wg), wg[0].shape[1]
    dX, dprob, dW = oracle.backward_all(x, dy, W, H, I, E, ids, p, L.token_routes, act=act)
    X = _f(x)
    DY = _f(dy)
    G = {e: _f(wg[e]) for e in range(E)}
    U = {e: _f(wu[e]) for e in range(E)}
    D = {e: _f(wd[e]) for e in range(E)}
    P = p.astype(np.float64)
    eps = 1e-4
    rng = np.random.default_rng(100 + seed)

    def num(fn_plus, fn_minus):
        return (fn_plus() - fn_minus()) / (2 * eps)

    def check(got, want, scale):
        assert abs(got - want) <= 2e-3 * max(scale, 1e-3), (got, want)

    sc = np.abs(dX).max()
    for _ in range(6):
        t, h = rng.integers(N), rng.integers(H)
        Xp, Xm = X.copy(), X.copy()
        Xp[t, h] += eps
        Xm[t, h] -= eps
        check(dX[t, h], num(lambda: _loss64(Xp, G, U, D, ids, P, DY, act),
                            lambda: _loss64(Xm, G, U, D, ids, P, DY, act)), sc)
    for name, Wd_ in (("g", G), ("u", U), ("d", D)):
        for _ in range(4):
            e = int(rng.integers(E))
            shape = Wd_[e].shape
            i, j = rng.integers(shape[0]), rng.integers(shape[1])
            Wp = {k: v.copy() for k, v in Wd_.items()}
            Wm = {k: v.copy() for k, v in Wd_.items()}
            Wp[e][i, j] += eps
            Wm[e][i, j] -= eps
            args_p = dict(g=G, u=U, d=D)
            args_m = dict(g=G, u=U, d=D)
            args_p[name] = Wp
            args_m[name] = Wm
            want = num(lambda: _loss64(X, args_p["g"], args_p["u"], args_p["d"], ids, P, DY, act),
                       lambda: _loss64(X, args_m["g"], args_m["u"], args_m["d"], ids, P, DY, act))
            got = {"d": dW[e][0], "g": dW[e][1], "u": dW[e][2]}[name][i, j]
            check(got, want, max(np.abs(dW[e][0]).max(), np.abs(dW[e][1]).max()))
    for _ in range(6):
        t, k = rng.integers(N), rng.integers(ids.shape[1])
        Pp, Pm = P.copy(), P.copy()
        Pp[t, k] += eps
        Pm[t, k] -= eps
        check(dprob[t, k], num(lambda: _loss64(X, G, U, D, ids, Pp, DY, act),
                               lambda: _loss64(X, G, U, D, ids, Pm, DY, act)), np.abs(dprob).max())


def test_weight_gradients_match_fp64_closed_form():
    x, dy, wg, wu, wd, ids, p, L, W = _problem(7, N=20, H=24, E=4, K=2, I=16)
    N, H = x.shape
    E, I = len(wg), wg[0].shape[1]
    _, _, dW = oracle.backward_all(x, dy, W, H, I, E, ids, p, L.token_routes)
    X, DY = _f(x), _f(dy)
    for e in range(E):
        dwd = np.zeros((I, H))
        dwg = np.zeros((H, I))
        dwu = np.zeros((H, I))
        for t in range(N):
            for k in range(ids.shape[1]):
                if ids[t, k] != e:
                    continue
                g = X[t] @ _f(wg[e])
                u = X[t] @ _f(wu[e])
                s = 1 / (1 + np.exp(-g))
                a = g * s * u
                dA = p[t, k] * (DY[t] @ _f(wd[e]).T)
                dwd += np.outer(p[t, k] * a, DY[t])
                dwg += np.outer(X[t], dA * u * s * (1 + g * (1 - s)))
                dwu += np.outer(X[t], dA * g * s)
        for got, want in zip(dW[e], (dwd, dwg, dwu)):
            assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())
