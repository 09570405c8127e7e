"""Shared set-up for the GPU parity tests: seeded inputs on the device, the
library's forward through the C ABI, and tolerance checks against the oracle."""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

import mixture_experts_routing_gb300 as moe
import oracle
import synth
import synth.gpu

# BF16 outputs against the fp32 oracle: max-abs error and relative Frobenius error.
TOL_MAX_ABS = 2e-2
TOL_REL_FRO = 1e-2


def bf16_dev(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str) -> None:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.size == 0:
        return
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= TOL_MAX_ABS and rel <= TOL_REL_FRO, "%s: max-abs %.3g rel-fro %.3g" % (what, err, rel)


def assert_close_intermediate(got: np.ndarray, ref: np.ndarray, what: str) -> None:
    """Tolerance for the bf16 intermediates h and o (the stated max-abs 2e-2
    applies to the layer output y). Each element is rounded to bf16 once
    (error <= 2^-8 of its magnitude); o also inherits h's rounding through a
    sum of I random-signed terms, a few 0.1 % of the row's RMS. Bound:
    |got-ref| <= 2^-7*|ref| + 0.02*rms(ref), and relative Frobenius <= 1e-2."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.size == 0:
        return
    d = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    worst = (d - 2.0 ** -7 * np.abs(ref)).max() / max(rms, 1e-30)
    assert rel <= TOL_REL_FRO and worst <= 0.02, "%s: rel-fro %.3g, excess %.3g rms" % (what, rel, worst)


class Problem:
    """One workload's inputs on the device plus the library's buffers."""

    def __init__(self, w: synth.Workload, bm: int = 32, dev="cuda:0", host_weights: bool = True,
                 bias: Optional[np.ndarray] = None, renorm: int = 1, x_bits: Optional[np.ndarray] = None,
                 with_ffn: bool = True, activation: int = 0, prob_in_act: int = 0):
        self.w, self.bm, self.dev = w, bm, torch.device(dev)
        N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
        self.activation, self.prob_in_act = activation, prob_in_act
        self.cfg = moe.Config(N, H, E, K, I, w.cap_num, w.cap_den, block_m=bm, renorm=renorm,
                              ladder=list(w.ladder), ladder_den=w.ladder_den,
                              activation=activation, prob_in_act=prob_in_act)
        self.x_bits = (x_bits if x_bits is not None
                       else synth.normal_bf16_bits(w.seed, synth.STREAM["x"], 0, N * H, w.x_std).reshape(N, H))
        self.wr = synth.normal_f32(w.seed, synth.STREAM["wr"], 0, H * E, w.wr_std).reshape(H, E)
        if bias is None:
            bias = synth.router_bias(w)
        self.bias = bias
        self.x = bf16_dev(self.x_bits, self.dev) if N > 0 else torch.empty((1, H), dtype=torch.bfloat16, device=self.dev)
        self.wr_d = torch.from_numpy(self.wr).to(self.dev)
        self.bias_d = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).to(self.dev)
        bf = dict(dtype=torch.bfloat16, device=self.dev)
        self.host_w: Dict[str, Dict[int, np.ndarray]] = {"wg": {}, "wu": {}, "wd": {}}
        self.with_ffn = with_ffn
        self.routes = moe.alloc_routes(self.cfg, self.dev)
        self.ws = moe.alloc_workspace(self.cfg, self.dev)
        if not with_ffn:
            return
        wg = torch.empty((E, H, I), **bf)
        wu = torch.empty((E, H, I), **bf)
        wd = torch.empty((E, I, H), **bf)
        if host_weights:
            hw = synth.make_host_inputs(w)
            for k in ("wg", "wu", "wd"):
                self.host_w[k] = hw[k]
            wg.copy_(bf16_dev(np.stack([hw["wg"][e] for e in range(E)]), self.dev))
            wu.copy_(bf16_dev(np.stack([hw["wu"][e] for e in range(E)]), self.dev))
            wd.copy_(bf16_dev(np.stack([hw["wd"][e] for e in range(E)]), self.dev))
        else:
            synth.gpu.fill(wg, w.seed, synth.STREAM["wg"], w.w_std)
            synth.gpu.fill(wu, w.seed, synth.STREAM["wu"], w.w_std)
            synth.gpu.fill(wd, w.seed, synth.STREAM["wd"], w.w_std)
        self.w13 = torch.empty((E, 2 * I, H), **bf)
        self.w2 = torch.empty((E, H, I), **bf)
        moe.pack_w13(self.cfg, wg, wu, self.w13)
        moe.pack_w2(self.cfg, wd, self.w2)
        del wg, wu, wd
        self.h, self.o, self.y = moe.alloc_buffers(self.cfg, self.dev)
        # poison outputs so unwritten rows show up
        for t in (self.h, self.o, self.y):
            t.fill_(float("nan"))

    def run(self) -> None:
        if not self.with_ffn:
            moe.route_align(self.cfg, self.x, self.wr_d, self.bias_d, self.routes, self.ws)
            torch.cuda.synchronize()
            return
        moe.forward(self.cfg, self.x, self.wr_d, self.bias_d, self.w13, self.w2, self.routes,
                    self.ws, self.h, self.o, self.y)
        torch.cuda.synchronize()
        assert moe.device_error() == 0

    def expert_weights(self, experts) -> oracle.ExpertWeights:
        w, E, H, I = self.w, self.w.n_experts, self.w.hidden, self.w.inter
        for e in experts:
            if e not in self.host_w["wg"]:
                self.host_w["wg"][e] = synth.normal_bf16_bits(w.seed, synth.STREAM["wg"], e * H * I, H * I, w.w_std).reshape(H, I)
                self.host_w["wu"][e] = synth.normal_bf16_bits(w.seed, synth.STREAM["wu"], e * H * I, H * I, w.w_std).reshape(H, I)
                self.host_w["wd"][e] = synth.normal_bf16_bits(w.seed, synth.STREAM["wd"], e * I * H, I * H, w.w_std).reshape(I, H)
        return oracle.ExpertWeights(E, self.host_w["wg"], self.host_w["wu"], self.host_w["wd"])

    def oracle_routing(self) -> oracle.Routing:
        w = self.w
        if w.cap_num == 0:
            return dropless_routing(self)
        return oracle.route(self.x_bits, self.wr, self.bias, w.n_experts, w.top_k, w.cap_num,
                            w.cap_den, self.bm, renorm=bool(self.cfg.renorm))

    def routes_np(self) -> dict:
        N = self.w.n_tokens
        out = {n: getattr(self.routes, n).cpu().numpy() for n, _ in moe.Routes.FIELDS}
        for n in ("topk_ids", "topk_p", "keep", "token_routes"):
            out[n] = out[n][:N]
        return out


def dropless_routing(P: "Problem") -> oracle.Routing:
    """Router plus the dropless, bucketed layout, in the shape of oracle.Layout
    (slot arrays over the whole allocated bound)."""
    w = P.w
    ids, p, _, _ = oracle.router(P.x_bits, P.wr, P.bias, w.top_k, renorm=bool(P.cfg.renorm))
    D = oracle.dropless_layout(ids, w.n_experts, P.bm, list(w.ladder), w.ladder_den)
    keep = np.ones(ids.shape, np.uint8)
    L = oracle.Layout(w.n_tokens, 0, keep, D.expert_counts, D.expert_counts, D.sorted_slot_ids,
                      D.expert_ids, D.block_start, D.num_tokens_post_padded, D.token_routes)
    return oracle.Routing(ids, p, L)


def assert_routing_equal(P: Problem, R: oracle.Routing) -> None:
    g = P.routes_np()
    L = R.layout
    S = len(L.sorted_slot_ids)
    assert np.array_equal(g["topk_ids"], R.topk_ids), "topk_ids"
    assert np.array_equal(g["topk_p"].view(np.int32), R.topk_p.view(np.int32)), "topk_p bits"
    assert np.array_equal(g["keep"], L.keep), "keep"
    assert np.array_equal(g["expert_counts"], L.expert_counts), "expert_counts"
    assert np.array_equal(g["kept_counts"], L.kept_counts), "kept_counts"
    assert np.array_equal(g["sorted_slot_ids"][:S], L.sorted_slot_ids), "sorted_slot_ids"
    assert np.array_equal(g["expert_ids"][:len(L.expert_ids)], L.expert_ids), "expert_ids"
    assert np.array_equal(g["block_start"], L.block_start), "block_start"
    assert int(g["num_tokens_post_padded"][0]) == L.num_tokens_post_padded, "num_tokens_post_padded"
    assert np.array_equal(g["token_routes"], L.token_routes), "token_routes"
    check_slot_prob(P, R)


def check_expert_slots(P: Problem, R: oracle.Routing, experts) -> None:
    """h and o of every kept slot of the given experts against the oracle FFN,
    and zeros in the padding rows below the 16-row granule."""
    L = R.layout
    H, I = P.w.hidden, P.w.inter
    W = P.expert_weights(experts)
    h = P.h.float().cpu().numpy()
    o = P.o.float().cpu().numpy()
    for e in experts:
        base, kept = int(L.block_start[e]) * P.bm, int(L.kept_counts[e])
        if kept == 0:
            continue
        toks = L.sorted_slot_ids[base:base + kept]
        o_ref, h_ref = oracle.ffn_routes(toks, [e] * kept, P.x_bits, W, H, I, want_h=True)
        assert_close_intermediate(h[base:base + kept], h_ref, "h of expert %d" % e)
        assert_close_intermediate(o[base:base + kept], o_ref, "o of expert %d" % e)
        pad_end = base + (kept + 15) // 16 * 16
        assert np.all(h[base + kept:pad_end] == 0) and np.all(o[base + kept:pad_end] == 0)


def check_combine_property(P: Problem, R: oracle.Routing) -> None:
    """y[t] equals the fp64 gather-combine of the library's own o rows."""
    o = P.o.float().cpu().numpy().astype(np.float64)
    y = P.y.float().cpu().numpy()
    tr = R.layout.token_routes
    p = R.topk_p.astype(np.float64)
    ref = np.zeros(y.shape)
    mag = np.zeros(y.shape)
    for k in range(tr.shape[1]):
        m = tr[:, k] >= 0
        ref[m] += p[m, k:k + 1] * o[tr[m, k]]
        mag[m] += np.abs(p[m, k:k + 1] * o[tr[m, k]])
    # bf16 rounding of the output (half an ulp: 2^-8 relative) plus fp32 accumulation
    assert np.all(np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * mag + 1e-30)


def assert_close_grad(got: np.ndarray, ref: np.ndarray, what: str) -> None:
    """fp32 gradients of large magnitude: relative Frobenius <= 1e-2 and
    max-abs <= 2e-2 * max(1, max|ref|)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.size == 0:
        return
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    bound = TOL_MAX_ABS * max(1.0, np.abs(ref).max())
    assert rel <= TOL_REL_FRO and err <= bound, "%s: max-abs %.3g (bound %.3g) rel-fro %.3g" % (
        what, err, bound, rel)


class Backward:
    """Training forward (saving the pre-activations) and the expert-path
    backward of a Problem for a seeded dY, through the C ABI."""

    def __init__(self, P: Problem, dy_std: float = 1.0):
        w, dev = P.w, P.dev
        N, H, E, I, K = w.n_tokens, w.hidden, w.n_experts, w.inter, w.top_k
        S = max(moe.max_slots(P.cfg), 1)
        self.P = P
        self.dy_bits = synth.normal_bf16_bits(w.seed, synth.STREAM["dy"], 0, N * H, dy_std).reshape(N, H)
        self.dy = bf16_dev(self.dy_bits, dev) if N > 0 else torch.empty((1, H), dtype=torch.bfloat16, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.preact = torch.full((S, 2 * I), float("nan"), **bf)
        self.dx = torch.full((max(N, 1), H), float("nan"), **bf)
        self.dw13 = torch.full((E, 2 * I, H), float("nan"), dtype=torch.float32, device=dev)
        self.dw2 = torch.full((E, H, I), float("nan"), dtype=torch.float32, device=dev)
        self.dprob = torch.full((max(N, 1), K), float("nan"), dtype=torch.float32, device=dev)
        self.ws = moe.alloc_backward_workspace(P.cfg, dev)
        self.ws.fill_(0xFF)  # NaN bit patterns where a kernel reads before writing

    def run(self) -> None:
        P = self.P
        moe.route_align(P.cfg, P.x, P.wr_d, P.bias_d, P.routes, P.ws)
        moe.ffn_forward_train(P.cfg, P.routes, P.x, P.w13, P.w2, P.h, P.o, self.preact)
        moe.combine(P.cfg, P.routes, P.o, P.y)
        moe.ffn_backward(P.cfg, P.routes, P.x, P.w13, P.w2, self.preact, self.dy, self.dx,
                         self.dw13, self.dw2, self.dprob, self.ws)
        torch.cuda.synchronize()
        assert moe.device_error() == 0

    def weight_grads(self, e: int):
        """(dWd [I,H], dWg [H,I], dWu [H,I]) of expert e in the oracle's layout."""
        I = self.P.w.inter
        d13 = self.dw13[e].cpu().numpy()
        return self.dw2[e].cpu().numpy().T, d13[:I].T, d13[I:].T


def check_slot_prob(P: Problem, R: oracle.Routing) -> None:
    """slot_prob holds, bit for bit, p' of the route each slot holds, and 0 on
    every padding slot of the allocated bound."""
    g = P.routes_np()
    sp = g["slot_prob"][:len(R.layout.sorted_slot_ids)]  # the route list's S slots
    want = np.zeros(len(sp), np.float32)
    tr = R.layout.token_routes.ravel()
    r = np.nonzero(tr >= 0)[0]
    want[tr[r]] = R.topk_p.ravel()[r]
    assert np.array_equal(sp.view(np.int32), want.view(np.int32)), "slot_prob"
