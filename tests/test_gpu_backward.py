"""Expert-path backward on the GPU against the oracle: dX, dprob and the
weight gradients, in the dropless layout and in the capacity layout with
dropped routes, plus the saved pre-activations of the training forward."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (Backward, Problem, assert_close, assert_close_grad,
                      assert_close_intermediate, assert_routing_equal)

pytestmark = pytest.mark.gpu

SMALL = [
    # dropless, ladder; several experts, a few slot tiles each
    (synth.Workload("bwd_dl", 300, 256, 8, 3, 256, 0, 1, zipf_s=0.8, ladder=(2, 3, 4, 5, 6, 8),
                    ladder_den=4), 32),
    # dropless, one hot expert holding three 256-slot tiles; H = 128 (128-wide wgrad N tile)
    (synth.Workload("bwd_hot", 640, 128, 6, 2, 384, 0, 1, zipf_s=2.0, ladder=(1, 2), ladder_den=2), 16),
    # capacity layout with drops (F = 1/2), skewed routing
    (synth.Workload("bwd_cap", 512, 256, 16, 2, 256, 1, 2, zipf_s=1.5), 64),
]


def _check_all(B: Backward):
    P = B.P
    w = P.w
    N, H, E, I = w.n_tokens, w.hidden, w.n_experts, w.inter
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    W = P.expert_weights(range(E))
    dX, dprob, dW = oracle.backward_all(P.x_bits, B.dy_bits, W, H, I, E, R.topk_ids, R.topk_p,
                                        R.layout.token_routes)
    assert_close(B.dx.float().cpu().numpy()[:N], dX, "dX")
    dp = B.dprob.cpu().numpy()[:N]
    assert_close_grad(dp, dprob, "dprob")
    assert np.all(dp[R.layout.token_routes < 0] == 0), "dprob of dropped routes"
    for e in range(E):
        got = B.weight_grads(e)
        for name, g, r in zip(("dW_down", "dW_gate", "dW_up"), got, dW[e]):
            if int(R.layout.kept_counts[e]) == 0:
                assert np.all(g == 0), "%s of empty expert %d" % (name, e)
            else:
                assert_close_grad(g, r, "%s of expert %d" % (name, e))
    return R


@pytest.mark.parametrize("w,bm", SMALL, ids=[s[0].name for s in SMALL])
def test_backward_small_elementwise(w, bm):
    P = Problem(w, bm=bm, host_weights=True)
    B = Backward(P)
    B.run()
    R = _check_all(B)
    if w.cap_num != 0:
        assert (R.layout.keep == 0).any(), "the capacity case must drop routes"


def test_training_forward_saves_preactivations():
    w = SMALL[0][0]
    P = Problem(w, bm=32, host_weights=True)
    B = Backward(P)
    B.run()
    R = P.oracle_routing()
    L = R.layout
    I = w.inter
    P.expert_weights(range(w.n_experts))
    pre = B.preact.float().cpu().numpy()
    for e in range(w.n_experts):
        base, kept = int(L.block_start[e]) * P.bm, int(L.kept_counts[e])
        if kept == 0:
            continue
        X = synth.bf16_bits_to_f32(P.x_bits[L.sorted_slot_ids[base:base + kept]]).astype(np.float64)
        wg = synth.bf16_bits_to_f32(P.host_w["wg"][e]).astype(np.float64)
        wu = synth.bf16_bits_to_f32(P.host_w["wu"][e]).astype(np.float64)
        assert_close_intermediate(pre[base:base + kept, :I], X @ wg, "g of expert %d" % e)
        assert_close_intermediate(pre[base:base + kept, I:], X @ wu, "u of expert %d" % e)
        pad_end = base + (kept + 15) // 16 * 16
        assert np.all(pre[base + kept:pad_end] == 0)


def test_backward_empty_batch():
    w = synth.Workload("bwd_empty", 0, 128, 4, 2, 128, 0, 1, ladder=(1, 2), ladder_den=1)
    P = Problem(w, bm=32, host_weights=True)
    B = Backward(P)
    B.run()
    assert np.all(B.dw13.cpu().numpy() == 0) and np.all(B.dw2.cpu().numpy() == 0)


def test_backward_full_size_sampled():
    """Dropless N = 16384, H = 4096, E = 64, top-6, I = 1408: dX and dprob of
    sampled tokens, and the weight gradients of the coldest expert."""
    w = synth.WORKLOADS["dropless"]
    P = Problem(w, bm=32, host_weights=False)
    B = Backward(P)
    B.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    N, H, E, I, K = w.n_tokens, w.hidden, w.n_experts, w.inter, w.top_k
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(N, 12, replace=False))
    experts = sorted({int(e) for e in R.topk_ids[toks].ravel()})
    kc = R.layout.kept_counts
    cold = int(np.argmin(np.where(kc > 0, kc, 1 << 30)))
    W = P.expert_weights(sorted(set(experts) | {cold}))
    tk = np.repeat(toks, K)
    ex = R.topk_ids[toks].ravel()
    pr = R.topk_p[toks].ravel()
    out = oracle.bwd_routes(tk, ex, pr, P.x_bits, B.dy_bits, W, H, I)
    dX_ref = out["dxr"].reshape(len(toks), K, H).sum(1)
    assert_close(B.dx.float().cpu().numpy()[toks], dX_ref, "dX (sampled tokens)")
    assert_close_grad(B.dprob.cpu().numpy()[toks].ravel(), out["dprob"], "dprob (sampled tokens)")
    # coldest expert: every route it holds, in slot order
    base, kept = int(R.layout.block_start[cold]) * P.bm, int(kc[cold])
    st = R.layout.sorted_slot_ids[base:base + kept]
    sel_t, sel_k = np.nonzero(R.topk_ids[st] == cold)
    pe = R.topk_p[st[sel_t], sel_k]
    o2 = oracle.bwd_routes(st, np.full(kept, cold, np.int32), pe, P.x_bits, B.dy_bits, W, H, I)
    ref = oracle.wgrad_expert(st, P.x_bits, B.dy_bits, o2["aw"], o2["dg"], o2["du"], H, I)
    for name, g, r in zip(("dW_down", "dW_gate", "dW_up"), B.weight_grads(cold), ref):
        assert_close_grad(g, r, "%s of expert %d" % (name, cold))
