"""FP8 (E4M3, one fp32 scale per row) expert path on the GPU against the
oracle: the row quantiser bit for bit, FC1's h and FC2's o of every kept slot,
and the layer output y. The oracle chain quantises x and the weights itself
(its codes are checked equal to the GPU's first), rounds its fp32 h to bf16
as the path stores it, quantises that h, and runs FC2 and the combine; no
value it takes comes from the GPU."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_gb300 as moe
import oracle
import synth
from gpu_util import Problem, assert_close, assert_close_intermediate, assert_routing_equal

pytestmark = pytest.mark.gpu


def _q_dev(bits: np.ndarray, dev):
    m = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)
    rows, cols = bits.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    s = torch.empty(rows, dtype=torch.float32, device=dev)
    moe.quantize_rows_fp8(m, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _assert_same_codes(bits: np.ndarray, dev, what: str) -> None:
    q, s = _q_dev(bits, dev)
    qo, so = oracle.quantize_rows_fp8(bits)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32)), what + ": scales differ"
    bad = np.argwhere(q != qo)
    assert bad.size == 0, "%s: %d codes differ, first at %s (%#x vs %#x)" % (
        what, len(bad), bad[0], q[tuple(bad[0])], qo[tuple(bad[0])])


def test_quantize_rows_tie_saturation_and_subnormal_rows():
    """Rows whose largest magnitude is 448 have scale 1 exactly, so the codes
    are the format's own rounding of each value: ties to even, the subnormal
    range, both signs; plus a zero row, a row of equal values and a row whose
    scale is not a power of two."""
    vals = [448.0, 1.0625, 1.1875, -1.0625, -0.3, 2.0 ** -10, 3 * 2.0 ** -10, 0.75 * 2.0 ** -9,
            240.0, 232.0, -448.0, 0.0, 17.0, 19.0, 2.0 ** -7, 1e-30]
    rows = np.zeros((6, 64), np.float32)
    rows[0, :len(vals)] = vals
    rows[1, :len(vals)] = [-v for v in vals]
    rows[2] = 0.0                                  # all zero: scale 1, codes 0
    rows[3] = 3.25                                 # every value the amax
    rows[4] = np.linspace(-5.0, 7.0, 64)           # scale 7/448
    rows[5, ::2] = 1e-3
    rows[5, 1::2] = -2e-3
    _assert_same_codes(synth.f32_to_bf16_bits(rows), torch.device("cuda:0"), "hand rows")


# widths that take each form of the quantiser: one warp per row holding 2, 4
# or 8 groups per lane, 2, 4 or 8 warps per row, and two passes above 16384
@pytest.mark.parametrize("rows,cols,std", [(37, 256, 1.0), (1000, 7168, 0.02), (8, 8, 50.0),
                                           (300, 1408, 3.0), (5, 1024, 1.0), (17, 2048, 1.0),
                                           (40, 4096, 1.0), (9, 12288, 0.5), (3, 16392, 2.0)])
def test_quantize_rows_random_bit_exact(rows, cols, std):
    rng = np.random.default_rng(rows + cols)
    m = (rng.standard_normal((rows, cols)) * std).astype(np.float32)
    m[rows // 2] = 0.0
    _assert_same_codes(synth.f32_to_bf16_bits(m), torch.device("cuda:0"), "%dx%d" % (rows, cols))


@pytest.mark.parametrize("cols,bound", [(128, 6), (4096, 5), (12288, 3)])
def test_quantize_rows_device_row_bound(cols, bound):
    """Rows at or past the device-side bound keep their contents; the rows
    below it equal the oracle's codes (also when the bound falls inside a CTA
    whose rows span several warps)."""
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(9)
    bits = synth.f32_to_bf16_bits(rng.standard_normal((10, cols)).astype(np.float32))
    m = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    q = torch.full((10, cols), 0xAB, dtype=torch.uint8, device=dev)
    s = torch.full((10,), -1.0, dtype=torch.float32, device=dev)
    bd = torch.tensor([bound], dtype=torch.int32, device=dev)
    moe.quantize_rows_fp8(m, q, s, rows_dev=bd)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_rows_fp8(bits[:bound])
    assert np.array_equal(q[:bound].cpu().numpy(), qo)
    assert np.array_equal(s[:bound].cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert bool((q[bound:] == 0xAB).all()) and bool((s[bound:] == -1.0).all())


def test_quantize_rows_rejects_bad_arguments():
    dev = torch.device("cuda:0")
    m = torch.zeros((4, 12), dtype=torch.bfloat16, device=dev)  # cols not a multiple of 8
    q = torch.empty((4, 12), dtype=torch.uint8, device=dev)
    s = torch.empty(4, dtype=torch.float32, device=dev)
    with pytest.raises(moe.MoEError):
        moe.quantize_rows_fp8(m, q, s)


class Fp8Problem:
    """A Problem whose expert path runs on FP8 operands."""

    def __init__(self, w, act: int = 0, pia: int = 0, host_weights: bool = True):
        self.P = P = Problem(w, bm=32, host_weights=host_weights, activation=act, prob_in_act=pia)
        self.wq = moe.Fp8Weights(P.cfg, P.w13, P.w2)
        self.xq, self.xs, self.hq, self.hs = moe.alloc_fp8_buffers(P.cfg, P.dev)

    def run(self) -> None:
        P = self.P
        moe.route_align(P.cfg, P.x, P.wr_d, P.bias_d, P.routes, P.ws)
        moe.ffn_forward_fp8(P.cfg, P.routes, P.x, self.wq, self.xq, self.xs, P.h, self.hq,
                            self.hs, P.o)
        moe.combine(P.cfg, P.routes, P.o, P.y)
        torch.cuda.synchronize()
        assert moe.device_error() == 0


def _packed_bits(P: Problem, e: int):
    """Host bf16 bits of expert e's packed w13 [2I, H] and w2 [H, I] rows,
    transposed from the seeded per-expert weights."""
    W = P.expert_weights([e])
    wg, wu, wd = P.host_w["wg"][e], P.host_w["wu"][e], P.host_w["wd"][e]
    del W
    return (np.ascontiguousarray(np.concatenate([wg.T, wu.T], 0)), np.ascontiguousarray(wd.T))


def _oracle_routes(P: Problem, e: int, toks, probs, xq, xs, check_weights: bool):
    """Oracle h (fp32) and o (fp32) of routes of expert e for tokens toks
    (rows of xq/xs); the weights' codes are checked against the GPU's."""
    w = P.w
    H, I = w.hidden, w.inter
    w13_bits, w2_bits = _packed_bits(P, e)
    w13q, w13s = oracle.quantize_rows_fp8(w13_bits)
    w2q, w2s = oracle.quantize_rows_fp8(w2_bits)
    if check_weights:
        assert np.array_equal(w13q, P._fp8.wq.w13q[e].cpu().numpy()), "w13 codes of expert %d" % e
        assert np.array_equal(w13s.view(np.uint32),
                              P._fp8.wq.w13_scale[e * 2 * I:(e + 1) * 2 * I].cpu().numpy().view(np.uint32))
        assert np.array_equal(w2q, P._fp8.wq.w2q[e].cpu().numpy()), "w2 codes of expert %d" % e
    n = len(toks)
    h = oracle.fc1_fp8_routes(np.asarray(toks, np.int32), np.zeros(n, np.int32), xq, xs,
                              w13q[None], w13s[None], H, I, act=P.activation,
                              scales=(np.asarray(probs, np.float32) if P.prob_in_act else None))
    hq, hs = oracle.quantize_rows_fp8(synth.f32_to_bf16_bits(h))
    o = oracle.fc2_fp8_routes(np.zeros(n, np.int32), hq, hs, w2q[None], w2s[None], H, I)
    return h, o


CASES = [
    (synth.WORKLOADS["tiny"], 0, 0),
    (synth.WORKLOADS["tiny"], 1, 1),
    (synth.WORKLOADS["qwen3_small"], 0, 0),
    (synth.Workload("fp8_dl", 300, 256, 8, 3, 256, 0, 1, zipf_s=0.8, ladder=(2, 3, 4, 5, 6, 8),
                    ladder_den=4), 1, 0),
    (synth.Workload("fp8_cap", 700, 384, 12, 3, 384, 1, 2, zipf_s=1.2), 0, 1),
]


@pytest.mark.parametrize("w,act,pia", CASES,
                         ids=["%s-act%d-pia%d" % (c[0].name, c[1], c[2]) for c in CASES])
def test_fp8_forward_elementwise(w, act, pia):
    F = Fp8Problem(w, act, pia)
    P = F.P
    P._fp8 = F
    F.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    # x codes: the GPU's equal the oracle's
    xq, xs = oracle.quantize_rows_fp8(P.x_bits)
    assert np.array_equal(F.xq.cpu().numpy()[:N], xq)
    assert np.array_equal(F.xs.cpu().numpy()[:N].view(np.uint32), xs.view(np.uint32))
    L = R.layout
    h = P.h.float().cpu().numpy()
    o = P.o.float().cpu().numpy()
    o_routes = np.zeros((N, K, H), np.float32)
    slot_of = L.token_routes
    for e in range(E):
        base, kept = int(L.block_start[e]) * P.bm, int(L.kept_counts[e])
        if kept == 0:
            continue
        toks = L.sorted_slot_ids[base:base + kept]
        ks = [int(np.nonzero(slot_of[t] == base + j)[0][0]) for j, t in enumerate(toks)]
        probs = [R.topk_p[t, k] for t, k in zip(toks, ks)]  # the oracle's p' of each slot
        h_ref, o_ref = _oracle_routes(P, e, toks, probs, xq, xs, check_weights=True)
        assert_close_intermediate(h[base:base + kept], h_ref, "h of expert %d" % e)
        assert_close_intermediate(o[base:base + kept], o_ref, "o of expert %d" % e)
        for j, (t, k) in enumerate(zip(toks, ks)):
            o_routes[t, k] = o_ref[j]
    y_ref = oracle.combine(0, N, L.keep, None if pia else R.topk_p, o_routes)
    y = P.y.float().cpu().numpy()[:N]
    assert_close(y, y_ref, "y")
    # the FP8 path stays near the bf16 layer: E4M3 carries 3 mantissa bits
    # (relative step 2^-3, error up to 2^-4 per element), averaged over the
    # contractions
    W = P.expert_weights(range(E))
    y_bf16 = oracle.forward_tokens(0, N, P.x_bits, W, H, I, R.topk_ids, R.topk_p, L.keep, act=act,
                                   prob_in_act=bool(pia))
    rel = np.linalg.norm(y - y_bf16) / max(np.linalg.norm(y_bf16), 1e-30)
    assert rel < 0.1, "FP8 vs bf16 layer: rel-fro %.3g" % rel


def test_fp8_h_quantised_consistently():
    """The path's own quantisation of h: for every kept slot, the decoded
    codes times the row scale stay within half an E4M3 step of h, and the
    scale is amax/448 (decoded with torch's float8_e4m3fn)."""
    w = synth.WORKLOADS["qwen3_small"]
    F = Fp8Problem(w)
    P = F.P
    F.run()
    R = P.oracle_routing()
    L = R.layout
    h = P.h.float().cpu()
    dq = F.hq.cpu().view(torch.float8_e4m3fn).float() * F.hs.cpu()[:, None]
    for e in range(w.n_experts):
        base, kept = int(L.block_start[e]) * P.bm, int(L.kept_counts[e])
        if kept == 0:
            continue
        hr, dr = h[base:base + kept], dq[base:base + kept]
        amax = hr.abs().amax(dim=1)
        sc = F.hs.cpu()[base:base + kept]
        assert torch.equal(sc, torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)))
        assert bool(((dr - hr).abs() <= 2.0 ** -4 * hr.abs() + 2.0 ** -10 * sc[:, None]).all())


def test_fp8_forward_full_size_sampled_tokens():
    """DeepSeek-V3 layer shape (4096 tokens, H 7168, 256 experts, top-8, I
    2048, capacity 1.25): whole tokens through the oracle's FP8 chain for a
    sample of tokens (every kept route of each)."""
    w = synth.WORKLOADS["dsv3"]
    F = Fp8Problem(w, host_weights=False)
    P = F.P
    P._fp8 = F
    F.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    N, H, K = w.n_tokens, w.hidden, w.top_k
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(N, 3, replace=False))
    xq, xs = oracle.quantize_rows_fp8(P.x_bits[toks])
    L = R.layout
    by_expert = {}
    for i, t in enumerate(toks):
        for k in range(K):
            if L.keep[t, k]:
                by_expert.setdefault(int(R.topk_ids[t, k]), []).append((i, k))
    o_routes = np.zeros((len(toks), K, H), np.float32)
    for n, (e, routes) in enumerate(sorted(by_expert.items())):
        rows = [i for i, _ in routes]
        probs = [R.topk_p[toks[i], k] for i, k in routes]
        _, o = _oracle_routes(P, e, rows, probs, xq, xs, check_weights=(n < 2))
        for (i, k), orow in zip(routes, o):
            o_routes[i, k] = orow
    y = P.y.float().cpu().numpy()
    for i, t in enumerate(toks):
        ref = oracle.combine(int(t), int(t) + 1, L.keep, R.topk_p, o_routes[i:i + 1])
        assert_close(y[t:t + 1], ref, "y of token %d" % t)
