"""Graph bucket ladder on the GPU: a replay of a bucket's captured forward on
n tokens computes the oracle's layer on those n tokens (routing bit-exact up
to the sentinel value, y within the stated tolerance) and equals an eager
forward on exactly those n tokens (y bit-identical), for capacity and
dropless layouts; eager fallback past the padding ratio; new inputs between
replays ("[4/5] feat: capture the FFN experts at bucketed padded shapes",
What this adds and Testing)."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_gb300 as moe
import oracle
import synth
import synth.gpu
from gpu_util import assert_close, bf16_dev

pytestmark = pytest.mark.gpu


def _layer(w, seed=0):
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    dev = torch.device("cuda:0")
    cfg = moe.Config(N, H, E, K, I, w.cap_num, w.cap_den, block_m=32, ladder=list(w.ladder),
                     ladder_den=w.ladder_den)
    wr = torch.from_numpy(synth.normal_f32(seed, synth.STREAM["wr"], 0, H * E, w.wr_std).reshape(H, E)).to(dev)
    b = synth.router_bias(w) if seed == w.seed else synth.zipf_bias(seed, E, w.zipf_s)
    bias = None if b is None else torch.from_numpy(b).to(dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    wg, wu, wd = torch.empty((E, H, I), **bf), torch.empty((E, H, I), **bf), torch.empty((E, I, H), **bf)
    synth.gpu.fill(wg, seed, synth.STREAM["wg"], w.w_std)
    synth.gpu.fill(wu, seed, synth.STREAM["wu"], w.w_std)
    synth.gpu.fill(wd, seed, synth.STREAM["wd"], w.w_std)
    w13, w2 = torch.empty((E, 2 * I, H), **bf), torch.empty((E, H, I), **bf)
    moe.pack_w13(cfg, wg, wu, w13)
    moe.pack_w2(cfg, wd, w2)
    return cfg, wr, bias, w13, w2


def _eager(w, n, x, wr, bias, w13, w2):
    """Forward on exactly n tokens (its own buffers)."""
    dev = x.device
    c = moe.Config(n, w.hidden, w.n_experts, w.top_k, w.inter, w.cap_num, w.cap_den, block_m=32,
                   ladder=list(w.ladder), ladder_den=w.ladder_den)
    r = moe.alloc_routes(c, dev)
    ws = moe.alloc_workspace(c, dev)
    h, o, y = moe.alloc_buffers(c, dev)
    xn = x[:max(n, 1)].contiguous()
    moe.forward(c, xn, wr, bias, w13, w2, r, ws, h, o, y)
    torch.cuda.synchronize()
    return y[:n].clone(), {k: getattr(r, k).cpu().numpy() for k, _ in moe.Routes.FIELDS}, moe.max_slots(c)


def _check_equal(L, n, w, y_e, r_e, s_e, bucket):
    assert torch.equal(L.y[:n].view(torch.int16), y_e.view(torch.int16)), "y (n=%d)" % n
    g = {k: getattr(L.routes, k).cpu().numpy() for k, _ in moe.Routes.FIELDS}
    K = w.top_k
    for k in ("topk_ids", "topk_p", "keep", "token_routes"):
        assert np.array_equal(g[k][:n].view(np.int32) if k == "topk_p" else g[k][:n],
                              r_e[k][:n].view(np.int32) if k == "topk_p" else r_e[k][:n]), k
        if n < bucket:  # rows in [n, bucket) are absent from the replayed batch
            tail = g[k][n:bucket]
            assert np.all(tail == (0 if k in ("topk_p", "keep") else -1)), k + " past n"
    for k in ("expert_counts", "kept_counts", "block_start", "num_tokens_post_padded"):
        assert np.array_equal(g[k], r_e[k]), k
    ssi_g, ssi_e = g["sorted_slot_ids"][:s_e].copy(), r_e["sorted_slot_ids"][:s_e].copy()
    ssi_g[ssi_g == bucket] = -7  # the sentinel is the bucket in a replay, n in the eager call
    ssi_e[ssi_e == n] = -7
    assert np.array_equal(ssi_g, ssi_e), "sorted_slot_ids"
    assert np.array_equal(g["slot_prob"][:s_e].view(np.int32), r_e["slot_prob"][:s_e].view(np.int32))


CAP = synth.Workload("ladder_cap", 2048, 512, 16, 4, 512, 5, 4, zipf_s=0.7)
DL = synth.Workload("ladder_dl", 2048, 512, 16, 4, 512, 0, 1, zipf_s=0.8, ladder=(2, 3, 4, 6, 8),
                    ladder_den=4)


@pytest.mark.parametrize("w", [CAP, DL], ids=["capacity", "dropless"])
def test_ladder_replay_equals_eager(w):
    cfg, wr, bias, w13, w2 = _layer(w)
    buckets = [128, 256, 512, 1024, 2048]
    L = moe.Ladder(cfg, buckets, 0.0, wr, bias, w13, w2, "cuda:0")
    xb = synth.normal_bf16_bits(7, synth.STREAM["x"], 0, w.n_tokens * w.hidden, 1.0).reshape(w.n_tokens, w.hidden)
    L.x.copy_(bf16_dev(xb, L.x.device))
    for n in (1, 100, 128, 129, 300, 1000, 1500, 2047, 2048):
        b = L.forward(n)
        torch.cuda.synchronize()
        assert b == next(i for i, v in enumerate(buckets) if v >= n)
        y_e, r_e, s_e = _eager(w, n, L.x, wr, bias, w13, w2)
        _check_equal(L, n, w, y_e, r_e, s_e, buckets[b])
    assert moe.device_error() == 0
    L.close()


def _host_weights(w):
    H, I = w.hidden, w.inter
    wg, wu, wd = {}, {}, {}
    for e in range(w.n_experts):
        wg[e] = synth.normal_bf16_bits(w.seed, synth.STREAM["wg"], e * H * I, H * I, w.w_std).reshape(H, I)
        wu[e] = synth.normal_bf16_bits(w.seed, synth.STREAM["wu"], e * H * I, H * I, w.w_std).reshape(H, I)
        wd[e] = synth.normal_bf16_bits(w.seed, synth.STREAM["wd"], e * I * H, I * H, w.w_std).reshape(I, H)
    return oracle.ExpertWeights(w.n_experts, wg, wu, wd)


def _oracle_layer(w, xb, wr, bias, n, bm=32):
    """The oracle's routing (fields in the library's naming) and y for the
    first n tokens as one batch."""
    E, K = w.n_experts, w.top_k
    xs = xb[:n]
    if w.cap_num == 0:
        ids, p, _, _ = oracle.router(xs, wr, bias, K)
        D = oracle.dropless_layout(ids, E, bm, list(w.ladder), w.ladder_den)
        keep = np.ones(ids.shape, np.uint8)
        lay = dict(expert_counts=D.expert_counts, kept_counts=D.expert_counts,
                   block_start=D.block_start, sorted_slot_ids=D.sorted_slot_ids,
                   expert_ids=D.expert_ids, ntpp=D.num_tokens_post_padded,
                   token_routes=D.token_routes)
    else:
        R = oracle.route(xs, wr, bias, E, K, w.cap_num, w.cap_den, bm)
        ids, p, keep, L = R.topk_ids, R.topk_p, R.layout.keep, R.layout
        lay = dict(expert_counts=L.expert_counts, kept_counts=L.kept_counts,
                   block_start=L.block_start, sorted_slot_ids=L.sorted_slot_ids,
                   expert_ids=L.expert_ids, ntpp=L.num_tokens_post_padded,
                   token_routes=L.token_routes)
    lay.update(topk_ids=ids, topk_p=p, keep=keep)
    return lay


@pytest.mark.parametrize("w", [CAP, DL], ids=["capacity", "dropless"])
def test_ladder_replay_matches_oracle(w):
    """Each replay's routing bit for bit, and y elementwise, against the
    oracle run on the n live tokens alone (capacity and ladder extents
    follow n)."""
    cfg, wr, bias, w13, w2 = _layer(w)
    buckets = [128, 256, 512, 1024, 2048]
    L = moe.Ladder(cfg, buckets, 0.0, wr, bias, w13, w2, "cuda:0")
    xb = synth.normal_bf16_bits(11, synth.STREAM["x"], 0, w.n_tokens * w.hidden, 1.0).reshape(w.n_tokens, w.hidden)
    L.x.copy_(bf16_dev(xb, L.x.device))
    wr_h = wr.cpu().numpy()
    bias_h = None if bias is None else bias.cpu().numpy()
    W = _host_weights(w)
    bm = 32
    for n in (1, 100, 129, 1500, 2048):
        b = L.forward(n)
        torch.cuda.synchronize()
        bucket = buckets[b]
        ref = _oracle_layer(w, xb, wr_h, bias_h, n, bm)
        g = {k: getattr(L.routes, k).cpu().numpy() for k, _ in moe.Routes.FIELDS}
        for k in ("topk_ids", "keep", "token_routes"):
            assert np.array_equal(g[k][:n], ref[k]), "%s (n=%d)" % (k, n)
        assert np.array_equal(g["topk_p"][:n].view(np.int32), ref["topk_p"].view(np.int32)), n
        for k in ("expert_counts", "kept_counts", "block_start"):
            assert np.array_equal(g[k], ref[k]), "%s (n=%d)" % (k, n)
        ntpp = int(g["num_tokens_post_padded"][0])
        assert ntpp == ref["ntpp"], n
        ssi = g["sorted_slot_ids"][:ntpp].copy()
        ssi_ref = ref["sorted_slot_ids"][:ntpp].copy()
        # the sentinel is the bucket in a replay, n in the oracle
        assert np.array_equal(ssi == bucket, ssi_ref == n), "sentinel slots (n=%d)" % n
        live = ssi_ref != n
        assert np.array_equal(ssi[live], ssi_ref[live]), "sorted_slot_ids (n=%d)" % n
        assert np.array_equal(g["expert_ids"][:ntpp // bm], ref["expert_ids"][:ntpp // bm]), n
        y_ref = oracle.forward_tokens(0, n, xb[:n], W, w.hidden, w.inter, ref["topk_ids"],
                                      ref["topk_p"], ref["keep"])
        assert_close(L.y[:n].float().cpu().numpy(), y_ref, "y (n=%d, bucket %d)" % (n, bucket))
    assert moe.device_error() == 0
    L.close()


def test_ladder_eager_fallback_and_new_inputs():
    w = CAP
    cfg, wr, bias, w13, w2 = _layer(w)
    buckets = [256, 512, 1024, 2048]
    L = moe.Ladder(cfg, buckets, 1.5, wr, bias, w13, w2, "cuda:0")
    for it, (n, want_b) in enumerate([(300, -1), (400, 1), (1500, 3), (100, -1), (256, 0)]):
        xb = synth.normal_bf16_bits(20 + it, synth.STREAM["x"], 0, w.n_tokens * w.hidden, 1.0)
        L.x.copy_(bf16_dev(xb.reshape(w.n_tokens, w.hidden), L.x.device))  # new input each time
        b = L.forward(n)
        torch.cuda.synchronize()
        assert b == want_b
        y_e, r_e, s_e = _eager(w, n, L.x, wr, bias, w13, w2)
        assert torch.equal(L.y[:n].view(torch.int16), y_e.view(torch.int16)), "y (n=%d)" % n
    L.close()


def test_ladder_empty_batch():
    w = DL
    cfg, wr, bias, w13, w2 = _layer(w)
    L = moe.Ladder(cfg, [512, 2048], 0.0, wr, bias, w13, w2, "cuda:0")
    assert L.forward(0) == 0
    torch.cuda.synchronize()
    assert int(L.routes.num_tokens_post_padded.item()) == 0
    assert np.all(L.routes.topk_ids.cpu().numpy()[:512] == -1)
    assert moe.device_error() == 0
    L.close()
