"""Router backward on the GPU against the oracle: dW_r, dbias and the router
path of dX for a seeded dprob, with and without renormalisation, including
the accumulation into an existing dX and the full-size shapes."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_gb300 as moe
import oracle
import synth
from gpu_util import Problem, assert_close, assert_close_grad, bf16_dev

pytestmark = pytest.mark.gpu


def _run(P, dprob, dx0_bits=None):
    w = P.w
    N, H, E = w.n_tokens, w.hidden, w.n_experts
    dev = P.dev
    moe.route_align(P.cfg, P.x, P.wr_d, P.bias_d, P.routes, P.ws)
    dx = (bf16_dev(dx0_bits, dev) if dx0_bits is not None
          else torch.zeros((max(N, 1), H), dtype=torch.bfloat16, device=dev))
    dwr = torch.full((H, E), float("nan"), dtype=torch.float32, device=dev)
    dbias = torch.full((E,), float("nan"), dtype=torch.float32, device=dev)
    ws = moe.alloc_router_backward_workspace(P.cfg, dev)
    dp = torch.from_numpy(np.ascontiguousarray(dprob, np.float32)).to(dev) if N > 0 else \
        torch.zeros((1, w.top_k), dtype=torch.float32, device=dev)
    moe.router_backward(P.cfg, P.routes, P.x, P.wr_d, P.bias_d, dp, dx, dwr, dbias, ws)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    return dx.float().cpu().numpy()[:N], dwr.cpu().numpy(), dbias.cpu().numpy()


SMALL = [
    (synth.Workload("rb_tiny", 256, 128, 8, 2, 128, 1, 1), 1),
    (synth.Workload("rb_norenorm", 300, 256, 8, 3, 128, 1, 1, zipf_s=1.0), 0),
    (synth.Workload("rb_e64", 520, 256, 64, 6, 128, 0, 1, zipf_s=0.8, ladder=(2, 4), ladder_den=2), 1),
    (synth.Workload("rb_e256", 333, 384, 256, 8, 128, 5, 4), 1),
    # E not a multiple of 4: W_r rows are not 16-byte multiples
    (synth.Workload("rb_e6", 200, 128, 6, 2, 128, 1, 1, zipf_s=0.5), 1),
    # experts padded to 128 and to 192 split columns (three 64-wide chunks)
    (synth.Workload("rb_e100", 257, 256, 100, 4, 128, 1, 1), 1),
    (synth.Workload("rb_e160", 190, 128, 160, 6, 128, 5, 4), 1),
    # many token splits of dW_r, the last one 8 tokens long
    (synth.Workload("rb_splits", 5000, 512, 64, 6, 128, 0, 1), 1),
    # fewer tokens than one tensor-map box (64 rows for dW_r, 128 for dx)
    (synth.Workload("rb_n5", 5, 128, 8, 2, 128, 1, 1), 1),
    (synth.Workload("rb_n40", 40, 256, 64, 4, 128, 1, 1), 1),
]


@pytest.mark.parametrize("w,renorm", SMALL, ids=[s[0].name for s in SMALL])
def test_router_backward_small_elementwise(w, renorm):
    P = Problem(w, bm=32, renorm=renorm, with_ffn=False)
    rng = np.random.default_rng(11)
    dprob = rng.standard_normal((w.n_tokens, w.top_k)).astype(np.float32)
    dx, dwr, dbias = _run(P, dprob)
    ref = oracle.router_backward(P.x_bits, P.wr, P.bias, w.top_k, dprob, renorm=bool(renorm))
    assert np.array_equal(P.routes.topk_ids.cpu().numpy()[:w.n_tokens], ref["topk_ids"])
    assert_close_grad(dwr, ref["dwr"], "dW_r")
    assert_close_grad(dbias, ref["dbias"], "dbias")
    assert_close(dx, ref["dx"], "router dX")


def test_router_backward_accumulates_into_dx():
    w = SMALL[0][0]
    P = Problem(w, bm=32, with_ffn=False)
    rng = np.random.default_rng(12)
    dprob = rng.standard_normal((w.n_tokens, w.top_k)).astype(np.float32)
    dx0 = synth.f32_to_bf16_bits(rng.standard_normal((w.n_tokens, w.hidden)).astype(np.float32))
    dx, _, _ = _run(P, dprob, dx0)
    ref = oracle.router_backward(P.x_bits, P.wr, P.bias, w.top_k, dprob)
    want = synth.bf16_bits_to_f32(dx0).astype(np.float64) + ref["dx"]
    assert_close(dx, want, "dX + router dX")
    # one rounding of the fp32 sum: within half a bf16 ulp of the exact sum
    assert np.all(np.abs(dx - want) <= 2.0 ** -8 * np.abs(want) + 1e-6)


@pytest.mark.parametrize("name", ["dsv3", "dropless"])
def test_router_backward_full_size(name):
    w = synth.WORKLOADS[name]
    P = Problem(w, bm=32, with_ffn=False)
    rng = np.random.default_rng(13)
    dprob = rng.standard_normal((w.n_tokens, w.top_k)).astype(np.float32)
    dx, dwr, dbias = _run(P, dprob)
    ref = oracle.router_backward(P.x_bits, P.wr, P.bias, w.top_k, dprob, want_dx=False)
    assert_close_grad(dwr, ref["dwr"], "dW_r")
    assert_close_grad(dbias, ref["dbias"], "dbias")
    # router dX of sampled tokens: dl (oracle) . W_r^T in fp64
    toks = np.sort(rng.choice(w.n_tokens, 16, replace=False))
    want = ref["dlogits"][toks].astype(np.float64) @ P.wr.T.astype(np.float64)
    assert_close(dx[toks], want, "router dX (sampled tokens)")


def test_router_backward_empty_batch():
    w = synth.Workload("rb_empty", 0, 128, 8, 2, 128, 1, 1)
    P = Problem(w, bm=32, with_ffn=False)
    _, dwr, dbias = _run(P, np.zeros((0, 2), np.float32))
    assert np.all(dwr == 0) and np.all(dbias == 0)


@pytest.mark.parametrize("w", [SMALL[2][0], synth.WORKLOADS["qwen3_30b"]], ids=["e64", "qwen3_30b"])
def test_router_backward_with_forward_logits_is_bit_identical(w):
    """The logits route_align left in its workspace give exactly the outputs
    of the recomputed ones."""
    P = Problem(w, bm=32, host_weights=True, with_ffn=False)
    N, H, E, K = w.n_tokens, w.hidden, w.n_experts, w.top_k
    dev = P.dev
    moe.route_align(P.cfg, P.x, P.wr_d, P.bias_d, P.routes, P.ws)
    rng = np.random.default_rng(4)
    dp = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32)).to(dev)
    ws = moe.alloc_router_backward_workspace(P.cfg, dev)
    outs = []
    for logits in (None, moe.route_workspace_logits(P.cfg, P.ws)):
        dx = torch.zeros((N, H), dtype=torch.bfloat16, device=dev)
        dwr = torch.full((H, E), float("nan"), dtype=torch.float32, device=dev)
        dbias = torch.full((E,), float("nan"), dtype=torch.float32, device=dev)
        moe.router_backward(P.cfg, P.routes, P.x, P.wr_d, P.bias_d, dp, dx, dwr, dbias, ws,
                            logits=logits)
        torch.cuda.synchronize()
        outs.append((dx.view(torch.int16).cpu(), dwr.view(torch.int32).cpu(),
                     dbias.view(torch.int32).cpu()))
    assert moe.device_error() == 0
    for a, b in zip(*outs):
        assert torch.equal(a, b)
