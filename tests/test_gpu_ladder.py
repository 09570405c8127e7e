"""Graph bucket ladder on the GPU: a replay of a bucket's captured forward on
n tokens equals an eager forward on exactly those n tokens (y bit-identical,
routing identical up to the sentinel value), for capacity and dropless
layouts; eager fallback past the padding ratio; new inputs between replays."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_gb300 as moe
import synth
import synth.gpu
from gpu_util import bf16_dev

pytestmark = pytest.mark.gpu


def _layer(w, seed=0):
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    dev = torch.device("cuda:0")
    cfg = moe.Config(N, H, E, K, I, w.cap_num, w.cap_den, block_m=32, ladder=list(w.ladder),
                     ladder_den=w.ladder_den)
    wr = torch.from_numpy(synth.normal_f32(seed, synth.STREAM["wr"], 0, H * E, w.wr_std).reshape(H, E)).to(dev)
    bias = None if w.zipf_s is None else torch.from_numpy(synth.zipf_bias(seed, E, w.zipf_s)).to(dev)
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
