"""Pins of the oracle's router backward (the gradient of the routing
probabilities p' through top-K renormalisation and the softmax, then to W_r,
the bias and x). Central finite differences in fp64 of the router written with
numpy (the chosen experts held fixed: the top-K selection is piecewise
constant), and the invariants of the softmax backward. No GPU."""
import numpy as np
import pytest

import oracle
import synth


def _f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _loss64(X, Wr, b, ids, dprob, renorm):
    """L = sum_{t,k} dprob[t,k] * p'[t,k] in fp64, the chosen experts fixed."""
    l = X @ Wr + (0.0 if b is None else b)
    l = l - l.max(1, keepdims=True)
    p = np.exp(l)
    p /= p.sum(1, keepdims=True)
    pk = np.take_along_axis(p, ids, 1)
    if renorm:
        pk = pk / pk.sum(1, keepdims=True)
    return float((dprob * pk).sum())


def _problem(seed, N=10, H=12, E=6, K=3):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    wr = (rng.standard_normal((H, E)) * 0.5).astype(np.float32)
    b = (rng.standard_normal(E) * 0.3).astype(np.float32)
    dprob = rng.standard_normal((N, K)).astype(np.float32)
    return x, wr, b, dprob


@pytest.mark.parametrize("seed,renorm", [(0, True), (1, False), (2, True)])
def test_router_backward_matches_central_differences(seed, renorm):
    x, wr, b, dprob = _problem(seed)
    N, H = x.shape
    E, K = wr.shape[1], dprob.shape[1]
    o = oracle.router_backward(x, wr, b, K, dprob, renorm=renorm)
    ids = o["topk_ids"]
    X, W, B = _f64(x), wr.astype(np.float64), b.astype(np.float64)
    D = dprob.astype(np.float64)
    eps = 1e-5
    rng = np.random.default_rng(50 + seed)

    def fd(fplus, fminus):
        return (fplus() - fminus()) / (2 * eps)

    def close(got, want, scale):
        assert abs(got - want) <= 1e-3 * max(scale, 1e-6), (got, want)

    # d L / d logits: perturb one logit of one token
    for _ in range(8):
        t, e = int(rng.integers(N)), int(rng.integers(E))

        l = X @ W + B

        def loss_l(dl):
            ll = l.copy()
            ll[t, e] += dl
            ll = ll - ll.max(1, keepdims=True)
            p = np.exp(ll)
            p /= p.sum(1, keepdims=True)
            pk = np.take_along_axis(p, ids, 1)
            if renorm:
                pk = pk / pk.sum(1, keepdims=True)
            return float((D * pk).sum())
        close(o["dlogits"][t, e], (loss_l(eps) - loss_l(-eps)) / (2 * eps), np.abs(o["dlogits"]).max())
    for _ in range(6):
        h, e = int(rng.integers(H)), int(rng.integers(E))
        Wp, Wm = W.copy(), W.copy()
        Wp[h, e] += eps
        Wm[h, e] -= eps
        close(o["dwr"][h, e], fd(lambda: _loss64(X, Wp, B, ids, D, renorm),
                                 lambda: _loss64(X, Wm, B, ids, D, renorm)), np.abs(o["dwr"]).max())
    for e in range(E):
        Bp, Bm = B.copy(), B.copy()
        Bp[e] += eps
        Bm[e] -= eps
        close(o["dbias"][e], fd(lambda: _loss64(X, W, Bp, ids, D, renorm),
                                lambda: _loss64(X, W, Bm, ids, D, renorm)), np.abs(o["dbias"]).max())
    for _ in range(6):
        t, h = int(rng.integers(N)), int(rng.integers(H))
        Xp, Xm = X.copy(), X.copy()
        Xp[t, h] += eps
        Xm[t, h] -= eps
        close(o["dx"][t, h], fd(lambda: _loss64(Xp, W, B, ids, D, renorm),
                                lambda: _loss64(Xm, W, B, ids, D, renorm)), np.abs(o["dx"]).max())


def test_router_backward_invariants():
    x, wr, b, dprob = _problem(3, N=40, H=16, E=8, K=2)
    o = oracle.router_backward(x, wr, b, 2, dprob)
    # the softmax backward sums to zero over the experts of a token
    assert np.abs(o["dlogits"].sum(1)).max() <= 1e-6 * max(1.0, np.abs(o["dlogits"]).max())
    # with renormalisation, a dprob constant over k changes nothing: sum_k p'_k = 1
    c = np.repeat(np.linspace(-1, 1, 40, dtype=np.float32)[:, None], 2, axis=1)
    oc = oracle.router_backward(x, wr, b, 2, c)
    assert np.abs(oc["dlogits"]).max() <= 1e-7
    # dbias is the column sum of dlogits, dx and dW_r the two products with it
    assert np.allclose(o["dbias"], o["dlogits"].astype(np.float64).sum(0), atol=1e-6)
    X = _f64(x)
    assert np.allclose(o["dwr"], X.T @ o["dlogits"].astype(np.float64), atol=1e-5)
    assert np.allclose(o["dx"], o["dlogits"].astype(np.float64) @ wr.T.astype(np.float64), atol=1e-5)


def test_router_backward_k_equals_e_without_renorm_is_softmax_jacobian():
    """K = E, no renormalisation: p' are the softmax probabilities (in expert
    order of the top-K), so dl = (diag(p) - p p^T) g with g the dprob of each
    expert: the softmax Jacobian written out in fp64."""
    x, wr, b, _ = _problem(4, N=6, H=10, E=5, K=5)
    rng = np.random.default_rng(9)
    dprob = rng.standard_normal((6, 5)).astype(np.float32)
    o = oracle.router_backward(x, wr, b, 5, dprob, renorm=False)
    ids, p = o["topk_ids"], o["probs"].astype(np.float64)
    for t in range(6):
        g = np.zeros(5)
        g[ids[t]] = dprob[t]
        J = np.diag(p[t]) - np.outer(p[t], p[t])
        assert np.allclose(o["dlogits"][t], J @ g, atol=1e-6)
