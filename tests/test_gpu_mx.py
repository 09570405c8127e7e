"""MX block-scaled FP8 (MXFP8 E4M3: an E8M0 scale per 32 values along the
contraction) expert path on the GPU against the oracle: the quantiser's codes
and scale bytes bit for bit (plain and in the GEMMs' atom layout), FC1's h
and FC2's o of every kept slot, and the layer output y. The oracle chain
quantises x and the weights itself (its codes are checked equal to the GPU's
first), rounds its fp32 h to bf16 as the path stores it, quantises that h,
and runs FC2 and the combine; no value it takes comes from the GPU."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_gb300 as moe
import oracle
import synth
from gpu_util import Problem, assert_close, assert_close_intermediate, assert_routing_equal

pytestmark = pytest.mark.gpu


def to_atoms(sc: np.ndarray) -> np.ndarray:
    """Plain [rows, cols/32] scale bytes to the 512-byte atom layout the MX
    GEMMs read (rows and cols multiples of 128)."""
    rows, nb = sc.shape
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    idx = ((r // 128) * (nb // 4) + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + b % 4
    out = np.zeros(rows * nb, np.uint8)
    out[idx.ravel()] = sc.ravel()
    return out


def _bf16_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _q_dev(bits: np.ndarray, dev, atoms=False):
    m = _bf16_dev(bits, dev)
    rows, cols = bits.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if atoms:
        s = torch.empty(rows * cols // 32, dtype=torch.uint8, device=dev)
        moe.quantize_mx_fp8_weights(m, q, s)
    else:
        s = torch.empty((rows, cols // 32), dtype=torch.uint8, device=dev)
        moe.quantize_mx_fp8(m, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _assert_same(bits: np.ndarray, dev, what: str, atoms=False) -> None:
    q, s = _q_dev(bits, dev, atoms)
    qo, so = oracle.quantize_mx_fp8(bits)
    want_s = to_atoms(so) if atoms else so
    assert np.array_equal(s, want_s), what + ": scale bytes differ"
    bad = np.argwhere(q != qo)
    assert bad.size == 0, "%s: %d codes differ, first at %s (%#x vs %#x)" % (
        what, len(bad), bad[0], q[tuple(bad[0])], qo[tuple(bad[0])])


def test_quantize_mx_hand_blocks():
    """Blocks whose maximum is a power of two times 448 or 256 (exact scaled
    values), ties of the E4M3 rounding, saturation (block maximum in
    [448, 512) times the scale), subnormal codes, all-zero blocks, both signs,
    and the clamped scale of tiny blocks."""
    rows = np.zeros((4, 256), np.float32)
    vals = [448.0, 1.0625, 1.1875, -1.0625, -0.3, 2.0 ** -10, 3 * 2.0 ** -10, 0.75 * 2.0 ** -9,
            240.0, 232.0, -448.0, 0.0, 17.0, 19.0, 2.0 ** -7, 1e-30]
    rows[0, :16] = vals                          # scale 2^0
    rows[0, 32:48] = [v * 2.0 ** -20 for v in vals]  # same block shape at 2^-20
    rows[0, 64:96] = 500.0                       # saturates: 500 * 2^0 > 448
    rows[0, 96] = 511.0
    rows[1, :32] = np.linspace(-5.0, 7.0, 32)
    rows[1, 32:64] = 2.0 ** -130                 # scale clamped at 2^-127
    rows[2] = -3.25                              # every value the maximum
    rows[3, ::2] = 1e-3
    rows[3, 1::2] = -2e-3
    _assert_same(synth.f32_to_bf16_bits(rows), torch.device("cuda:0"), "hand blocks")


@pytest.mark.parametrize("rows,cols,std", [(37, 256, 1.0), (1000, 7168, 0.02), (8, 32, 50.0),
                                           (300, 1408, 3.0), (5, 96, 1.0), (17, 2048, 1.0)])
def test_quantize_mx_random_bit_exact(rows, cols, std):
    rng = np.random.default_rng(rows + cols)
    scale = np.exp2(rng.integers(-30, 30, size=(rows, 1)))
    m = (rng.standard_normal((rows, cols)) * std * scale).astype(np.float32)
    m[rows // 2] = 0.0
    _assert_same(synth.f32_to_bf16_bits(m), torch.device("cuda:0"), "%dx%d" % (rows, cols))


@pytest.mark.parametrize("rows,cols", [(128, 128), (512, 2048), (384, 7168)])
def test_quantize_mx_weight_atoms_bit_exact(rows, cols):
    rng = np.random.default_rng(rows)
    m = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    m[5] *= 1000.0
    _assert_same(synth.f32_to_bf16_bits(m), torch.device("cuda:0"), "atoms %dx%d" % (rows, cols),
                 atoms=True)


def test_quantize_mx_device_row_bound():
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(9)
    bits = synth.f32_to_bf16_bits(rng.standard_normal((10, 512)).astype(np.float32))
    m = _bf16_dev(bits, dev)
    q = torch.full((10, 512), 0xAB, dtype=torch.uint8, device=dev)
    s = torch.full((10, 16), 0xCD, dtype=torch.uint8, device=dev)
    bd = torch.tensor([6], dtype=torch.int32, device=dev)
    moe.quantize_mx_fp8(m, q, s, rows_dev=bd)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_mx_fp8(bits[:6])
    assert np.array_equal(q[:6].cpu().numpy(), qo) and np.array_equal(s[:6].cpu().numpy(), so)
    assert bool((q[6:] == 0xAB).all()) and bool((s[6:] == 0xCD).all())


def test_quantize_mx_rejects_bad_arguments():
    dev = torch.device("cuda:0")
    m = torch.zeros((4, 48), dtype=torch.bfloat16, device=dev)  # cols not a multiple of 32
    q = torch.empty((4, 48), dtype=torch.uint8, device=dev)
    s = torch.empty((4, 2), dtype=torch.uint8, device=dev)
    with pytest.raises(moe.MoEError):
        moe.quantize_mx_fp8(m, q, s)
    m2 = torch.zeros((100, 128), dtype=torch.bfloat16, device=dev)  # rows not a multiple of 128
    with pytest.raises(moe.MoEError):
        moe.quantize_mx_fp8_weights(m2, torch.empty((100, 128), dtype=torch.uint8, device=dev),
                                    torch.empty(400, dtype=torch.uint8, device=dev))


class MxProblem:
    """A Problem whose expert path runs on MX operands."""

    def __init__(self, w, act: int = 0, pia: int = 0, host_weights: bool = True):
        self.P = P = Problem(w, bm=32, host_weights=host_weights, activation=act, prob_in_act=pia)
        self.wq = moe.MxWeights(P.cfg, P.w13, P.w2)
        self.xq, self.xs, self.hq, self.hs = moe.alloc_mx_buffers(P.cfg, P.dev)

    def run(self) -> None:
        P = self.P
        moe.route_align(P.cfg, P.x, P.wr_d, P.bias_d, P.routes, P.ws)
        moe.ffn_forward_mx(P.cfg, P.routes, P.x, self.wq, self.xq, self.xs, P.h, self.hq, self.hs,
                           P.o)
        moe.combine(P.cfg, P.routes, P.o, P.y)
        torch.cuda.synchronize()
        assert moe.device_error() == 0


def _packed_bits(P: Problem, e: int):
    P.expert_weights([e])
    wg, wu, wd = P.host_w["wg"][e], P.host_w["wu"][e], P.host_w["wd"][e]
    return (np.ascontiguousarray(np.concatenate([wg.T, wu.T], 0)), np.ascontiguousarray(wd.T))


def _oracle_routes(F: MxProblem, e: int, toks, probs, xq, xs, check_weights: bool):
    """Oracle h and o (fp32) of routes of expert e for tokens toks (rows of
    xq/xs); the weights' codes and scale atoms are checked against the GPU's."""
    P = F.P
    w = P.w
    H, I = w.hidden, w.inter
    w13_bits, w2_bits = _packed_bits(P, e)
    w13q, w13s = oracle.quantize_mx_fp8(w13_bits)
    w2q, w2s = oracle.quantize_mx_fp8(w2_bits)
    if check_weights:
        n13, n2 = 2 * I * H // 32, H * I // 32
        assert np.array_equal(w13q, F.wq.w13q[e].cpu().numpy()), "w13 codes of expert %d" % e
        assert np.array_equal(to_atoms(w13s), F.wq.w13_sf[e * n13:(e + 1) * n13].cpu().numpy())
        assert np.array_equal(w2q, F.wq.w2q[e].cpu().numpy()), "w2 codes of expert %d" % e
        assert np.array_equal(to_atoms(w2s), F.wq.w2_sf[e * n2:(e + 1) * n2].cpu().numpy())
    n = len(toks)
    h = oracle.fc1_mx_routes(np.asarray(toks, np.int32), np.zeros(n, np.int32), xq, xs, w13q[None],
                             w13s, H, I, act=P.activation,
                             scales=(np.asarray(probs, np.float32) if P.prob_in_act else None))
    hq, hs = oracle.quantize_mx_fp8(synth.f32_to_bf16_bits(h))
    o = oracle.fc2_mx_routes(np.zeros(n, np.int32), hq, hs, w2q[None], w2s, H, I)
    return h, o


CASES = [
    (synth.WORKLOADS["tiny"], 0, 0),
    (synth.WORKLOADS["tiny"], 1, 1),
    (synth.WORKLOADS["qwen3_small"], 0, 0),
    (synth.Workload("mx_dl", 300, 256, 8, 3, 256, 0, 1, zipf_s=0.8, ladder=(2, 3, 4, 5, 6, 8),
                    ladder_den=4), 1, 0),
    (synth.Workload("mx_cap", 700, 384, 12, 3, 384, 1, 2, zipf_s=1.2), 0, 1),
    # ragged kept counts over several slot tiles of at most 224 slots
    (synth.Workload("mx_hot", 1200, 128, 4, 2, 128, 0, 1, zipf_s=2.0, ladder=(1, 2), ladder_den=2),
     0, 0),
]


@pytest.mark.parametrize("w,act,pia", CASES,
                         ids=["%s-act%d-pia%d" % (c[0].name, c[1], c[2]) for c in CASES])
def test_mx_forward_elementwise(w, act, pia):
    """The whole MX path: x codes bit for bit, h of every kept slot, and y
    against the oracle's MX chain at the stated tolerance. FC2 is then checked
    on its own with identical inputs: the oracle's bf16 h written into the
    slot rows, quantised and multiplied on the GPU, o of every kept slot
    against the oracle (the GPU's own h differs from the oracle's by bf16
    rounding in a few elements, and one such difference can move an E4M3 code
    by a whole step, so o is compared on the oracle's h)."""
    F = MxProblem(w, act, pia)
    P = F.P
    F.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    xq, xs = oracle.quantize_mx_fp8(P.x_bits)
    assert np.array_equal(F.xq.cpu().numpy()[:N], xq)
    assert np.array_equal(F.xs.cpu().numpy()[:N], xs)
    L = R.layout
    h = P.h.float().cpu().numpy()
    y = P.y.float().cpu().numpy()[:N]
    o_routes = np.zeros((N, K, H), np.float32)
    h_oracle = torch.zeros_like(P.h)  # the oracle's h, bf16, in slot order
    refs = {}
    for e in range(E):
        base, kept = int(L.block_start[e]) * P.bm, int(L.kept_counts[e])
        if kept == 0:
            continue
        toks = L.sorted_slot_ids[base:base + kept]
        ks = [int(np.nonzero(L.token_routes[t] == base + j)[0][0]) for j, t in enumerate(toks)]
        probs = [R.topk_p[t, k] for t, k in zip(toks, ks)]
        h_ref, o_ref = _oracle_routes(F, e, toks, probs, xq, xs, check_weights=True)
        assert_close_intermediate(h[base:base + kept], h_ref, "h of expert %d" % e)
        h_oracle[base:base + kept] = _bf16_dev(synth.f32_to_bf16_bits(h_ref), P.dev)
        refs[e] = (base, kept, o_ref)
        for j, (t, k) in enumerate(zip(toks, ks)):
            o_routes[t, k] = o_ref[j]
    y_ref = oracle.combine(0, N, L.keep, None if pia else R.topk_p, o_routes)
    assert_close(y, y_ref, "y")
    W = P.expert_weights(range(E))
    y_bf16 = oracle.forward_tokens(0, N, P.x_bits, W, H, I, R.topk_ids, R.topk_p, L.keep, act=act,
                                   prob_in_act=bool(pia))
    rel = np.linalg.norm(y - y_bf16) / max(np.linalg.norm(y_bf16), 1e-30)
    assert rel < 0.1, "MX vs bf16 layer: rel-fro %.3g" % rel
    # FC2 on the oracle's h
    P.o.fill_(float("nan"))
    moe.quantize_mx_fp8(h_oracle, F.hq, F.hs, rows_dev=P.routes.num_tokens_post_padded)
    moe.fc2_forward_mx(P.cfg, P.routes, F.hq, F.hs, F.wq.w2q, F.wq.w2_sf, P.o)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    o = P.o.float().cpu().numpy()
    for e, (base, kept, o_ref) in refs.items():
        assert_close_intermediate(o[base:base + kept], o_ref, "o of expert %d" % e)
        pad_end = base + (kept + 15) // 16 * 16
        assert np.all(o[base + kept:pad_end] == 0), "o padding of expert %d" % e


def test_mx_forward_full_size_sampled_tokens():
    """DeepSeek-V3 layer shape: whole tokens through the oracle's MX chain for
    a sample of tokens (every kept route of each)."""
    w = synth.WORKLOADS["dsv3"]
    F = MxProblem(w, host_weights=False)
    P = F.P
    F.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    N, H, K = w.n_tokens, w.hidden, w.top_k
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(N, 3, replace=False))
    xq, xs = oracle.quantize_mx_fp8(P.x_bits[toks])
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
        _, o = _oracle_routes(F, e, rows, probs, xq, xs, check_weights=(n < 2))
        for (i, k), orow in zip(routes, o):
            o_routes[i, k] = orow
    y = P.y.float().cpu().numpy()
    for i, t in enumerate(toks):
        ref = oracle.combine(int(t), int(t) + 1, L.keep, R.topk_p, o_routes[i:i + 1])
        assert_close(y[t:t + 1], ref, "y of token %d" % t)
