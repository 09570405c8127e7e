"""Activation variants on the GPU against the oracle: the GeGLU expert
activation (exact erf GELU) and the routing probability applied inside the
activation (unit-weight combine), forward and backward, and the route list's
per-slot probability."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (Backward, Problem, assert_close, assert_close_grad,
                      assert_close_intermediate, assert_routing_equal, check_slot_prob)

pytestmark = pytest.mark.gpu

CASES = [
    (synth.WORKLOADS["tiny"], 1, 0),
    (synth.WORKLOADS["tiny"], 0, 1),
    (synth.WORKLOADS["qwen3_small"], 1, 1),
    (synth.Workload("act_dl", 300, 256, 8, 3, 256, 0, 1, zipf_s=0.8, ladder=(2, 3, 4, 5, 6, 8),
                    ladder_den=4), 1, 1),
    (synth.Workload("act_cap", 700, 384, 12, 3, 384, 1, 2, zipf_s=1.2), 1, 0),
]


@pytest.mark.parametrize("w,act,pia", CASES,
                         ids=["%s-act%d-pia%d" % (c[0].name, c[1], c[2]) for c in CASES])
def test_forward_variants_elementwise(w, act, pia):
    P = Problem(w, bm=32, host_weights=True, activation=act, prob_in_act=pia)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    check_slot_prob(P, R)
    W = P.expert_weights(range(w.n_experts))
    y_ref = oracle.forward_tokens(0, w.n_tokens, P.x_bits, W, w.hidden, w.inter, R.topk_ids,
                                  R.topk_p, R.layout.keep, act=act, prob_in_act=bool(pia))
    assert_close(P.y.float().cpu().numpy()[:w.n_tokens], y_ref, "y")
    # h of every kept slot: act(g) u, times p' when the probability is in the activation
    L = R.layout
    h = P.h.float().cpu().numpy()
    sp = P.routes.slot_prob.cpu().numpy()
    for e in range(w.n_experts):
        base, kept = int(L.block_start[e]) * P.bm, int(L.kept_counts[e])
        if kept == 0:
            continue
        toks = L.sorted_slot_ids[base:base + kept]
        _, h_ref = oracle.ffn_routes(toks, [e] * kept, P.x_bits, W, w.hidden, w.inter, want_h=True,
                                     act=act, scales=sp[base:base + kept] if pia else None)
        assert_close_intermediate(h[base:base + kept], h_ref, "h of expert %d" % e)


@pytest.mark.parametrize("w", [CASES[3][0], CASES[4][0]], ids=["dropless", "capacity"])
def test_backward_geglu_elementwise(w):
    P = Problem(w, bm=32, host_weights=True, activation=1)
    B = Backward(P)
    B.run()
    R = P.oracle_routing()
    N, H, E, I = w.n_tokens, w.hidden, w.n_experts, w.inter
    W = P.expert_weights(range(E))
    dX, dprob, dW = oracle.backward_all(P.x_bits, B.dy_bits, W, H, I, E, R.topk_ids, R.topk_p,
                                        R.layout.token_routes, act=1)
    assert_close(B.dx.float().cpu().numpy()[:N], dX, "dX")
    assert_close_grad(B.dprob.cpu().numpy()[:N], dprob, "dprob")
    for e in range(E):
        if int(R.layout.kept_counts[e]) == 0:
            continue
        for name, g, r in zip(("dW_down", "dW_gate", "dW_up"), B.weight_grads(e), dW[e]):
            assert_close_grad(g, r, "%s of expert %d" % (name, e))


def test_forward_geglu_prob_in_act_full_size_tokens():
    """qwen3_30b shape with GeGLU and the probability in the activation: whole
    tokens through the oracle FFN (every kept route of the sampled tokens)."""
    w = synth.WORKLOADS["qwen3_30b"]
    P = Problem(w, bm=32, host_weights=False, activation=1, prob_in_act=1)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    check_slot_prob(P, R)
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(w.n_tokens, 6, replace=False))
    experts = sorted({int(e) for t in toks for e, k in zip(R.topk_ids[t], R.layout.keep[t]) if k})
    W = P.expert_weights(experts)
    y = P.y.float().cpu().numpy()
    for t in toks:
        ref = oracle.forward_tokens(int(t), int(t) + 1, P.x_bits, W, w.hidden, w.inter, R.topk_ids,
                                    R.topk_p, R.layout.keep, act=1, prob_in_act=True)
        assert_close(y[t:t + 1], ref, "y of token %d" % t)
