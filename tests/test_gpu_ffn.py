"""Expert FFN and combine on the GPU against the oracle (BF16 outputs within
max-abs 2e-2 and relative Frobenius 1e-2 of the fp32 oracle)."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_gb300 as moe
import oracle
import synth
from gpu_util import (Problem, assert_close, assert_routing_equal, check_combine_property,
                      check_expert_slots)

pytestmark = pytest.mark.gpu


def _w(N, H, E, K, I, cn=1, cd=1, **kw):
    return synth.Workload("case", N, H, E, K, I, cn, cd, **kw)


def _full_check(P):
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    w = P.w
    W = P.expert_weights(range(w.n_experts))
    y_ref = oracle.forward_tokens(0, w.n_tokens, P.x_bits, W, w.hidden, w.inter, R.topk_ids,
                                  R.topk_p, R.layout.keep)
    assert_close(P.y.float().cpu().numpy()[:w.n_tokens], y_ref, "y")
    check_expert_slots(P, R, range(w.n_experts))
    check_combine_property(P, R)
    return R


@pytest.mark.parametrize("name,bm", [("tiny", 32), ("tiny", 16), ("qwen3_small", 32),
                                     ("qwen3_small", 128)])
def test_forward_small_workloads_elementwise(name, bm):
    _full_check(Problem(synth.WORKLOADS[name], bm=bm, host_weights=True))


@pytest.mark.parametrize("w,bm", [
    (_w(300, 256, 6, 2, 384, cn=3, cd=4), 16),   # drops, ragged kept counts, 3 feature tiles
    (_w(700, 128, 4, 2, 256, cn=1, cd=1), 32),   # capacity 350: two slot tiles per expert, H=128
    (_w(129, 384, 3, 3, 128, cn=1, cd=1), 64),   # K = E, FC2 with an odd number of 128-row tiles
    (_w(40, 128, 16, 1, 128, cn=1, cd=4), 16),   # tiny capacity, many empty experts
    (_w(513, 512, 8, 2, 256, cn=2, cd=1), 128),  # capacity above the route count: no drops
])
def test_forward_random_shapes_elementwise(w, bm):
    _full_check(Problem(w, bm=bm, host_weights=True))


@pytest.mark.parametrize("name", ["qwen3_30b", "dsv3"])
def test_forward_full_size_sampled(name):
    """Full-size workload: routing bit-exact; h and o of every kept slot of
    three experts (the busiest, the emptiest non-empty, the median) against the
    oracle; y of every token as the gather-combine of the library's o."""
    w = synth.WORKLOADS[name]
    P = Problem(w, bm=32, host_weights=False)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    kc = R.layout.kept_counts
    order = np.argsort(kc, kind="stable")
    nonzero = [e for e in order if kc[e] > 0]
    experts = sorted({int(order[-1]), int(nonzero[0]), int(order[len(order) // 2])})
    check_expert_slots(P, R, experts)
    check_combine_property(P, R)
    dropped = ~R.layout.keep.any(1)
    if dropped.any():
        assert torch.all(P.y[torch.from_numpy(np.nonzero(dropped)[0]).to(P.dev)] == 0)


def test_forward_qwen3_30b_sampled_tokens_end_to_end():
    """A few whole tokens of the Zipf-routed workload through the oracle FFN,
    including one that lost routes to the capacity limit."""
    w = synth.WORKLOADS["qwen3_30b"]
    P = Problem(w, bm=32, host_weights=False)
    P.run()
    R = P.oracle_routing()
    keep = R.layout.keep
    partly = np.nonzero((keep.sum(1) > 0) & (keep.sum(1) < w.top_k))[0]
    toks = sorted({0, w.n_tokens - 1, int(partly[0]) if len(partly) else 1})
    experts = sorted({int(e) for t in toks for e in R.topk_ids[t]})
    W = P.expert_weights(experts)
    y = P.y.float().cpu().numpy()
    for t in toks:
        y_ref = oracle.forward_tokens(t, t + 1, P.x_bits, W, w.hidden, w.inter, R.topk_ids,
                                      R.topk_p, keep)
        assert_close(y[t:t + 1], y_ref, "y of token %d" % t)


def test_forward_dsv3_whole_tokens_and_spread_experts():
    """DeepSeek-V3-shaped layer at full size: whole tokens through the oracle
    layer (the first, the last, and tokens that lost a route to the capacity
    limit), and h and o of every kept slot of eight experts spread over the id
    range, so a wrong weight slice of any of them at H = 7168 shows."""
    w = synth.WORKLOADS["dsv3"]
    P = Problem(w, bm=32, host_weights=False)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    E = w.n_experts
    spread = sorted({int(e) for e in np.linspace(0, E - 1, 8).round()})
    check_expert_slots(P, R, spread)
    keep = R.layout.keep
    partly = np.nonzero((keep.sum(1) > 0) & (keep.sum(1) < w.top_k))[0]
    assert len(partly) > 0, "the workload is expected to drop some routes"
    toks = sorted({0, w.n_tokens - 1, int(partly[0]), int(partly[-1])})
    experts = sorted({int(e) for t in toks for e in R.topk_ids[t]})
    W = P.expert_weights(experts)
    y = P.y.float().cpu().numpy()
    for t in toks:
        y_ref = oracle.forward_tokens(t, t + 1, P.x_bits, W, w.hidden, w.inter, R.topk_ids,
                                      R.topk_p, keep)
        assert_close(y[t:t + 1], y_ref, "y of token %d" % t)


def test_empty_batch_is_a_no_op():
    P = Problem(_w(0, 128, 8, 2, 128), bm=16, host_weights=True)
    P.run()
    assert int(P.routes.num_tokens_post_padded.item()) == 0
    assert torch.all(P.routes.kept_counts == 0)


def test_pack_is_a_transpose():
    w = _w(16, 256, 3, 2, 384)
    P = Problem(w, bm=16, host_weights=True)
    for e in range(3):
        g = torch.from_numpy(P.host_w["wg"][e].view(np.int16)).view(torch.bfloat16)
        u = torch.from_numpy(P.host_w["wu"][e].view(np.int16)).view(torch.bfloat16)
        d = torch.from_numpy(P.host_w["wd"][e].view(np.int16)).view(torch.bfloat16)
        assert torch.equal(P.w13[e, :384].cpu(), g.t())
        assert torch.equal(P.w13[e, 384:].cpu(), u.t())
        assert torch.equal(P.w2[e].cpu(), d.t())


def test_graph_replay_equals_eager_with_new_inputs():
    """Capture the three calls once; replay with new token values of the same
    shape; every output equals an eager run on the same inputs."""
    w = synth.WORKLOADS["qwen3_small"]
    P = Problem(w, bm=32, host_weights=True)
    P.run()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            moe.forward(P.cfg, P.x, P.wr_d, P.bias_d, P.w13, P.w2, P.routes, P.ws, P.h, P.o, P.y)
    torch.cuda.synchronize()
    for seed in (11, 12):
        xb = synth.normal_bf16_bits(seed, 0, 0, w.n_tokens * w.hidden).reshape(w.n_tokens, w.hidden)
        P.x.copy_(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(P.dev))
        g.replay()
        torch.cuda.synchronize()
        got = {n: getattr(P.routes, n).clone() for n, _ in moe.Routes.FIELDS}
        y_graph = P.y.clone()
        o_graph = P.o.clone()
        P.run()
        for n, _ in moe.Routes.FIELDS:
            assert torch.equal(got[n], getattr(P.routes, n)), n
        S = int(P.routes.num_tokens_post_padded.item())
        kept = P.routes.token_routes[P.routes.token_routes >= 0].long()
        assert torch.equal(o_graph[kept], P.o[kept])
        assert torch.equal(y_graph, P.y)
        assert S == moe.max_slots(P.cfg)


@pytest.mark.parametrize("cn", [1, 0], ids=["capacity", "dropless"])
def test_forward_largest_token_count(cn):
    """The largest supported token count (24576) through the whole forward:
    routing bit-exact, every kept slot of the busiest and the emptiest
    non-empty expert against the oracle, y of every token as the combine of
    the library's o, and whole tokens (first, last, middle) end to end."""
    kw = dict(zipf_s=0.8, ladder=(2, 4), ladder_den=2) if cn == 0 else dict(zipf_s=0.8)
    w = synth.Workload("max_tokens", 24576, 256, 16, 4, 256, cn, 1, **kw)
    P = Problem(w, bm=32, host_weights=True)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    kc = R.layout.kept_counts
    order = np.argsort(kc, kind="stable")
    nonzero = [e for e in order if kc[e] > 0]
    check_expert_slots(P, R, sorted({int(order[-1]), int(nonzero[0])}))
    check_combine_property(P, R)
    toks = [0, w.n_tokens // 2, w.n_tokens - 1]
    W = P.expert_weights(range(w.n_experts))
    y = P.y.float().cpu().numpy()
    for t in toks:
        y_ref = oracle.forward_tokens(t, t + 1, P.x_bits, W, w.hidden, w.inter, R.topk_ids,
                                      R.topk_p, R.layout.keep)
        assert_close(y[t:t + 1], y_ref, "y of token %d" % t)
