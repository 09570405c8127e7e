"""Fits the stored router bias of the Zipf-skewed workloads.

TEST INFRASTRUCTURE: writes input data; it calls only the CPU oracle and the
seeded input generator, never the CUDA library.

The workloads that ask for Zipf(s) expert popularity (the Qwen3-30B-A3B-shaped
layer with s = 1.0, the dropless layer with s = 0.8) are given a per-expert
router bias b that makes the share of routes each expert receives follow the
target of ``synth.zipf_target_shares``: share of popularity rank r
proportional to r^-s, capped at 1/K (an expert holds at most one route per
token), summing to 1. Adding ``-s ln r`` alone does not do it: top-K selection
turns a softmax weight ratio into a much steeper route-share ratio at the head
and starves the tail.

Fit, on a calibration batch drawn from its own stream (``synth.STREAM
['xcal']``, never the x the tests and benchmark use), M tokens from the same
N(0,1) bf16 distribution, with the workload's own router weight W_r:

1. the oracle router gives the logits without bias, l0 = x . W_r (once);
2. start from b = -s ln(rank);
3. repeat: the routes of every token under logits l0 + b (the oracle adds the
   bias after the contraction, so these are its logits), top-K by logit
   (softmax keeps the order); realised share c_e / (M K); then
   b_e += eta ln(target_e / realised_e), damped; an expert whose target is
   the 1/K cap and that already takes nearly every token is left alone (its
   bias would otherwise grow without bound);
4. the result is checked with the oracle router itself (logits, softmax,
   top-K, ties to the lower expert) on the calibration batch, and reported on
   the first N tokens of the test stream.

The bias is defined up to a constant (softmax and top-K ignore it); it is
shifted so that the most popular expert's bias is 0.

Usage: python oracle/calibrate_router_bias.py qwen3_30b dropless dropless_e16
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def route_counts_by_logit(l0: np.ndarray, b: np.ndarray, K: int) -> np.ndarray:
    """Routes per expert when each token takes its K largest logits l0 + b."""
    l = l0 + b[None, :].astype(np.float32)
    top = np.argpartition(-l, K - 1, axis=1)[:, :K]
    return np.bincount(top.ravel(), minlength=l0.shape[1])


def fit(w: synth.Workload, m_tokens: int, iters: int, log=print):
    E, K, H = w.n_experts, w.top_k, w.hidden
    ranks = synth.zipf_ranks(w.seed, E)
    target = synth.zipf_target_shares(E, K, w.zipf_s)[ranks - 1]     # per expert
    capped = target >= (1.0 / K) * (1 - 1e-12)
    wr = synth.normal_f32(w.seed, synth.STREAM["wr"], 0, H * E, w.wr_std).reshape(H, E)
    xcal = synth.normal_bf16_bits(w.seed, synth.STREAM["xcal"], 0, m_tokens * H,
                                  w.x_std).reshape(m_tokens, H)
    t0 = time.time()
    _, _, _, l0 = oracle.router(xcal, wr, None, K, want_logits=True)
    log("%s: calibration logits of %d tokens in %.1f s" % (w.name, m_tokens, time.time() - t0))
    b = -w.zipf_s * np.log(ranks.astype(np.float64))
    R = m_tokens * K
    for it in range(iters):
        c = route_counts_by_logit(l0, b, K)
        real = np.maximum(c, 0.5) / R
        step = np.log(target / real)
        step[capped & (c >= 0.999 * m_tokens)] = 0.0
        eta = 0.7 if it < iters // 2 else 0.35
        b = b + eta * np.clip(step, -1.0, 1.0)
    b = b - b[np.argmin(ranks)]
    return b.astype(np.float32), ranks, target, wr, xcal


def shares(x_bits, wr, b, K, E):
    ids, _, _, _ = oracle.router(x_bits, wr, b, K)
    return np.bincount(ids.ravel(), minlength=E) / ids.size


def report(name, share, ranks, target, n_tokens, K, lines, log=print):
    by_rank = np.empty_like(share)
    by_rank[ranks - 1] = share
    t_rank = np.empty_like(target)
    t_rank[ranks - 1] = target
    rel = by_rank / t_rank - 1.0
    # binomial spread of a batch: an expert's count is a sum of N per-token
    # Bernoulli picks with probability K * share
    q = np.minimum(K * t_rank, 1.0)
    sigma = np.sqrt(n_tokens * q * (1 - q)) / (n_tokens * K * t_rank)
    within = int((np.abs(rel[:64]) <= 0.10).sum())
    head = " ".join("%.4f/%.4f" % (by_rank[r], t_rank[r]) for r in range(min(8, len(t_rank))))
    msg = ("%s: %d tokens; ranks 1-%d within 10%% of target: %d; max |rel. dev.| ranks 1-64 %.3f; "
           "max |dev.|/sigma %.2f; realised/target shares ranks 1-8: %s"
           % (name, n_tokens, min(64, len(t_rank)), within, float(np.abs(rel[:64]).max()),
              float(np.nanmax(np.abs(rel[:64]) / np.where(sigma[:64] > 0, sigma[:64], np.nan)))
              if (sigma[:64] > 0).any() else 0.0, head))
    log(msg)
    lines.append("# " + msg)
    return by_rank, rel


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("workloads", nargs="+")
    ap.add_argument("--tokens", type=int, default=65536, help="calibration batch size")
    ap.add_argument("--iters", type=int, default=300)
    a = ap.parse_args(argv)
    os.makedirs(os.path.dirname(synth.router_bias_path("x")), exist_ok=True)
    for name in a.workloads:
        w = synth.WORKLOADS[name]
        assert w.zipf_s is not None and w.calibrated_bias == name, name
        E, K = w.n_experts, w.top_k
        b, ranks, target, wr, xcal = fit(w, a.tokens, a.iters)
        lines = [
            "# Router bias of workload %r (%s)." % (name, w.note),
            "# Calibrated so that expert route shares follow Zipf(s=%g) capped at 1/K=1/%d:"
            % (w.zipf_s, K),
            "# %d calibration tokens of stream %d (not the x of tests and benchmark), %d"
            " fixed-point steps." % (a.tokens, synth.STREAM["xcal"], a.iters),
            "# Written by: python oracle/calibrate_router_bias.py %s" % name,
            "# Routes per expert checked with the oracle router:",
        ]
        report("calibration batch", shares(xcal, wr, b, K, E), ranks, target, a.tokens, K, lines)
        test_sizes = (w.n_tokens,) if not w.sweep else (w.sweep[-1],)
        for n in test_sizes:
            x = synth.normal_bf16_bits(w.seed, synth.STREAM["x"], 0, n * w.hidden,
                                       w.x_std).reshape(n, w.hidden)
            report("test batch", shares(x, wr, b, K, E), ranks, target, n, K, lines)
        lines.append("# expert  fp32 bits  (value, popularity rank)")
        for e in range(E):
            bits = int(np.array([b[e]], np.float32).view(np.uint32)[0])
            lines.append("%d %08x  # %.6f rank %d" % (e, bits, float(b[e]), int(ranks[e])))
        with open(synth.router_bias_path(name), "w") as f:
            f.write("\n".join(lines) + "\n")
        print("wrote", synth.router_bias_path(name))


if __name__ == "__main__":
    main()
