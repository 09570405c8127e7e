#!/usr/bin/env python3
"""MoE-layer forward benchmark on GB300.

One step = one forward of the whole layer over one batch of synthetic tokens:
moe_route_align (router, scan, drop-and-pad select, route-list layout), FC1
gather-GEMM + SwiGLU, FC2 grouped GEMM, gather-combine, each a C-ABI call.

Default workload: the DeepSeek-V3-shaped layer (N=4096 tokens, H=7168,
E=256, top-8, I=2048, F=1.25, ~22.5 GB of bf16 expert weights), the largest
workload that fits one GPU. Its inputs exceed L2, so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, on the host cores
    python bench.py --workload dropless    # training step of the dropless,
                                           # bucketed layer (forward + backward),
                                           # swept over N = 128 .. 16384
    python bench.py --mx                   # the same forward with MX block-scaled E4M3
                                           # expert GEMMs (E8M0 scale per 32 values)
    python bench.py --fp8                  # the same forward with the expert GEMMs
                                           # on E4M3 operands (row-wise scales): a
                                           # variant line; the headline is bf16
    python bench.py --serve [--workload qwen3_30b]
                                           # serving: a seeded sequence of
                                           # variable batch sizes through the
                                           # graph bucket ladder, and eager

Under torchrun each rank is an independent replica with its own batch (weak
scaling, no collective on the data path); value = tokens of all ranks / the
slowest rank's time. Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s on 1 GB300; grouped-GEMM TFLOPS as % of BF16 peak"
METRIC_SERVE = ("MoE-layer serving tokens/s on 1 GB300: seeded variable batch sizes through the "
                "graph bucket ladder")
METRIC_TRAIN = ("MoE-layer fwd+bwd tokens/s on 1 GB300 (dropless bucketed layer, dX/dW backward); "
                "TFLOPS as % of BF16 peak")
UNIT = "tokens/s"


# ----------------------------------------------------------------------------- helpers
def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3")
    ap.add_argument("--block-m", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="expert GEMMs on E4M3 operands with row-wise fp32 scales (x and h "
                         "quantised in the step); prints a variant line, not the bf16 headline")
    ap.add_argument("--mx", action="store_true",
                    help="expert GEMMs on MX block-scaled E4M3 operands (an E8M0 scale per 32 "
                         "values along the contraction); prints a variant line")
    ap.add_argument("--serve", action="store_true",
                    help="variable batch sizes through the graph bucket ladder")
    ap.add_argument("--serve-batches", type=int, default=64)
    ap.add_argument("--pad-ratio", type=float, default=0.0)
    ap.add_argument("--cpu-experts", type=int, default=48,
                    help="experts whose FFN the CPU baseline runs (bounded sample)")
    ap.add_argument("--activation", choices=["swiglu", "geglu"], default="swiglu",
                    help="gated activation of FC1 (forward and training steps)")
    ap.add_argument("--prob-in-act", action="store_true",
                    help="p' multiplies FC1's activation; the combine sums with unit weights")
    ap.add_argument("--no-extras", action="store_true",
                    help="default run only: skip the Qwen3-30B-shaped forward and the dropless "
                         "training step reported beside the headline")
    args = ap.parse_args(argv)
    if (args.fp8 or args.mx) and (args.activation != "swiglu" or args.prob_in_act):
        ap.error("--fp8 and --mx run the SwiGLU layer with p' in the combine")
    if args.fp8 and args.mx:
        ap.error("--fp8 (row scales) and --mx (block scales) are separate variants")
    return args


def act_code(args) -> int:
    """moe_config_t.activation (and the oracle's act): 0 SwiGLU, 1 GeGLU."""
    return 1 if args.activation == "geglu" else 0


def variant_config(args) -> dict:
    """Config keys of the activation variant (none for the default layer)."""
    d = {}
    if args.activation != "swiglu":
        d["activation"] = args.activation
    if args.prob_in_act:
        d["prob_in_act"] = True
    return d


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (the slowest rank's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "_source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["mixture_experts_routing_gb300/csrc/gemm.cu",
                "mixture_experts_routing_gb300/csrc/ptx.cuh"]


def ncu_traffic(kernel: str, workload: str, units: float):
    """DRAM bytes per launch from the committed ncu summary, scaled by the
    launch's units; None when absent or when the kernel changed since."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("workload") != workload:
        return None
    if d.get("source_hash") != source_hash(d.get("sources", GEMM_SOURCES)):
        return None
    return d["dram_bytes_per_unit"] * units


# ----------------------------------------------------------------------------- work model
def work_model(w, kept_counts, fp8=False, slots=0, mx=False):
    """Algorithmic bytes and flops per launch of each kernel, from the
    per-expert kept counts of this batch. fp8: GEMM operands are one byte
    (plus a 4-byte scale per row; with mx a one-byte scale per 32 values),
    and the two quantisation passes read bf16 x and the `slots` used rows of
    h."""
    import numpy as np
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    kc = np.asarray(kept_counts, dtype=np.int64)
    kept = int(kc.sum())
    active = int((kc > 0).sum())
    rows = int(((kc + 15) // 16 * 16).sum())  # slots the GEMMs compute (16-row granule)
    ob = (1.0 + 1.0 / 32 if mx else 1.0) if fp8 else 2.0  # bytes per GEMM operand element
    sb = 4.0 if fp8 and not mx else 0.0                    # bytes of scale per operand row
    m = {}
    m["fc1"] = {"flops": 2.0 * kept * H * 2 * I,
                "bytes": active * 2.0 * I * (H * ob + sb) + N * (H * ob + sb) + rows * I * 2,
                "units": active, "unit": "active expert"}
    m["fc2"] = {"flops": 2.0 * kept * I * H,
                "bytes": active * 1.0 * H * (I * ob + sb) + rows * (I * ob + sb) + rows * H * 2,
                "units": active, "unit": "active expert"}
    if fp8:
        m["quant_x"] = {"flops": 0.0, "bytes": N * H * (2.0 + ob) + N * sb, "units": N,
                        "unit": "token"}
        m["quant_h"] = {"flops": 0.0, "bytes": slots * I * (2.0 + ob) + slots * sb, "units": slots,
                        "unit": "slot"}
    m["combine"] = {"flops": 2.0 * kept * H, "bytes": kept * H * 2.0 + N * H * 2 + N * K * 8,
                    "units": N, "unit": "token"}
    m["route"] = {"flops": 2.0 * N * H * E, "bytes": N * H * 2.0 + H * E * 4 + N * E * 8 + N * K * 24,
                  "units": N, "unit": "token"}
    m["_kept"], m["_active"], m["_rows"] = kept, active, rows
    return m


def roofline_for(name, model, ms, peaks, workload, fp8=False, mx=False):
    """Roofline object of one kernel: bound, achieved, peak, frac, traffic.
    An E4M3 contraction takes the measured bf16 peak times the nominal
    FP8/BF16 dense ratio (4.5 / 2.25 PFLOP/s)."""
    d = model[name]
    sec = ms / 1e3
    hbm = peaks["hbm_gbs"]
    tensor = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    alu = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12  # fp32 FMA pipes
    if name == "route":
        t_c, peak_c = d["flops"] / (alu * 1e12), alu
    else:
        t_c, peak_c = d["flops"] / (tensor * 1e12), tensor
    t_m = d["bytes"] / (hbm * 1e9)
    src = peaks["_source"]
    if t_m >= t_c:
        ach = d["bytes"] / sec / 1e9
        r = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
             "peak_source": src, "frac_of_spec_8000_gbs": ach / 8000.0}
    else:
        ach = d["flops"] / sec / 1e12
        r = {"bound": "alu" if name == "route" else "tensor", "achieved": ach, "peak": peak_c,
             "unit": "TFLOP/s", "frac": ach / peak_c,
             "peak_source": src + (" x 2 (nominal FP8/BF16 ratio)" if fp8 and name != "route" else "")}
    tr = (ncu_traffic("moe_gemm_kernel:" + name + (("_mx" if mx else "_fp8") if fp8 else ""),
                      workload, d["units"])
          if name in ("fc1", "fc2") else None)
    r["traffic"] = tr
    r["kernel"] = name
    r["ms"] = ms
    r["algorithmic_bytes"] = d["bytes"]
    r["algorithmic_flops"] = d["flops"]
    return r


# ----------------------------------------------------------------------------- CPU oracle timing
def time_oracle_sample(w, x_bits, wr, bias, bm, n_experts_sample, seed_experts=0, act=0,
                       prob_in_act=False):
    """The oracle, as it stands, on a bounded sample of one step: routing of
    every token, expert FFN of `n_experts_sample` experts' kept routes
    (extrapolated to all kept routes by route count), combine of every token;
    act 0 SwiGLU / 1 GeGLU, prob_in_act: p' scales the activation and the
    combine has unit weights. Returns (tokens/s, description, seconds of CPU
    work, threads)."""
    import numpy as np
    import oracle
    import synth
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    t0 = time.perf_counter()
    R = oracle.route(x_bits, wr, bias, E, K, w.cap_num, w.cap_den, bm)
    t_route = time.perf_counter() - t0
    L = R.layout
    kept_total = int(L.kept_counts.sum())
    cand = [e for e in range(E) if L.kept_counts[e] > 0]
    rng = np.random.default_rng(seed_experts)
    sample = sorted(rng.choice(cand, size=min(n_experts_sample, len(cand)), replace=False).tolist())
    wg = {e: synth.normal_bf16_bits(w.seed, synth.STREAM["wg"], e * H * I, H * I, w.w_std).reshape(H, I) for e in sample}
    wu = {e: synth.normal_bf16_bits(w.seed, synth.STREAM["wu"], e * H * I, H * I, w.w_std).reshape(H, I) for e in sample}
    wd = {e: synth.normal_bf16_bits(w.seed, synth.STREAM["wd"], e * I * H, I * H, w.w_std).reshape(I, H) for e in sample}
    W = oracle.ExpertWeights(E, wg, wu, wd)
    toks, exps = [], []
    for e in sample:
        base = e * L.cpad
        k = int(L.kept_counts[e])
        toks += L.sorted_slot_ids[base:base + k].tolist()
        exps += [e] * k
    scales = None
    if prob_in_act:  # each route's p'
        ids = np.asarray(R.topk_ids)
        pk = np.asarray(R.topk_p)
        scales = np.array([pk[t][list(ids[t]).index(e)] for t, e in zip(toks, exps)], np.float32)
    t0 = time.perf_counter()
    oracle.ffn_routes(toks, exps, x_bits, W, H, I, act=act, scales=scales)
    t_ffn = time.perf_counter() - t0
    o_zero = np.zeros((N * K, H), dtype=np.float32)
    t0 = time.perf_counter()
    oracle.combine(0, N, L.keep, None if prob_in_act else R.topk_p, o_zero)
    t_comb = time.perf_counter() - t0
    t_full = t_route + t_ffn * kept_total / max(len(toks), 1) + t_comb
    desc = ("routing of all %d tokens + expert FFN of %d/%d experts (%d of %d kept routes, "
            "time extrapolated by route count) + combine of all tokens"
            % (N, len(sample), len(cand), len(toks), kept_total))
    return N / t_full, desc, t_route + t_ffn + t_comb, oracle.num_threads()


def time_oracle_sample_fp8(w, x_bits, wr, bias, bm, n_experts_sample, seed_experts=0, mx=False):
    """The oracle's FP8 chain (row scales; with mx block scales), as it
    stands, on a bounded sample of one step:
    routing and x quantisation of every token; FC1 on E4M3 operands, h
    rounded to bf16 and quantised, FC2 on E4M3 operands for the kept routes
    of `n_experts_sample` experts (extrapolated to all kept routes by route
    count; their weights are quantised once, outside the timing, as the GPU
    path does); combine of every token."""
    import numpy as np
    import oracle
    import synth
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    t0 = time.perf_counter()
    R = oracle.route(x_bits, wr, bias, E, K, w.cap_num, w.cap_den, bm)
    quant = oracle.quantize_mx_fp8 if mx else oracle.quantize_rows_fp8
    xq, xs = quant(x_bits)
    t_route = time.perf_counter() - t0
    L = R.layout
    kept_total = int(L.kept_counts.sum())
    cand = [e for e in range(E) if L.kept_counts[e] > 0]
    rng = np.random.default_rng(seed_experts)
    sample = sorted(rng.choice(cand, size=min(n_experts_sample, len(cand)), replace=False).tolist())
    t_ffn, n_routes = 0.0, 0
    for e in sample:
        wg = synth.normal_bf16_bits(w.seed, synth.STREAM["wg"], e * H * I, H * I, w.w_std).reshape(H, I)
        wu = synth.normal_bf16_bits(w.seed, synth.STREAM["wu"], e * H * I, H * I, w.w_std).reshape(H, I)
        wd = synth.normal_bf16_bits(w.seed, synth.STREAM["wd"], e * I * H, I * H, w.w_std).reshape(I, H)
        w13q, w13s = quant(np.ascontiguousarray(np.concatenate([wg.T, wu.T], 0)))
        w2q, w2s = quant(np.ascontiguousarray(wd.T))
        base, k = e * L.cpad, int(L.kept_counts[e])
        toks = L.sorted_slot_ids[base:base + k]
        zero = np.zeros(k, np.int32)
        t0 = time.perf_counter()
        if mx:
            h = oracle.fc1_mx_routes(toks, zero, xq, xs, w13q[None], w13s, H, I)
            hq, hs = quant(synth.f32_to_bf16_bits(h))
            oracle.fc2_mx_routes(zero, hq, hs, w2q[None], w2s, H, I)
        else:
            h = oracle.fc1_fp8_routes(toks, zero, xq, xs, w13q[None], w13s[None], H, I)
            hq, hs = quant(synth.f32_to_bf16_bits(h))
            oracle.fc2_fp8_routes(zero, hq, hs, w2q[None], w2s[None], H, I)
        t_ffn += time.perf_counter() - t0
        n_routes += k
    o_zero = np.zeros((N * K, H), dtype=np.float32)
    t0 = time.perf_counter()
    oracle.combine(0, N, L.keep, R.topk_p, o_zero)
    t_comb = time.perf_counter() - t0
    t_full = t_route + t_ffn * kept_total / max(n_routes, 1) + t_comb
    desc = ("%s chain: routing and x quantisation of all %d tokens + FC1/h quantisation/FC2 on "
            "E4M3 operands for %d/%d experts (%d of %d kept routes, time extrapolated by route "
            "count) + combine of all tokens" % ("MX" if mx else "FP8", N, len(sample), len(cand),
                                                n_routes, kept_total))
    return N / t_full, desc, t_route + t_ffn + t_comb, oracle.num_threads()


def host_inputs(w, rank_seed):
    import synth
    N, H, E = w.n_tokens, w.hidden, w.n_experts
    x_bits = synth.normal_bf16_bits(rank_seed, synth.STREAM["x"], 0, N * H, w.x_std).reshape(N, H)
    wr = synth.normal_f32(w.seed, synth.STREAM["wr"], 0, H * E, w.wr_std).reshape(H, E)
    bias = synth.router_bias(w)
    return x_bits, wr, bias


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    import synth
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    w = synth.WORKLOADS[args.workload]
    x_bits, wr, bias = host_inputs(w, w.seed)
    train = w.cap_num == 0
    dy_bits = None
    if train:
        dy_bits = synth.normal_bf16_bits(w.seed, synth.STREAM["dy"], 0, w.n_tokens * w.hidden,
                                         1.0).reshape(w.n_tokens, w.hidden)

    def sample(i, n):
        """One bounded sample on the first n tokens of the batch, taken as a
        batch of their own (per-token oracle work does not depend on N)."""
        wn, xn = w.with_tokens(n), x_bits[:n]
        if train:  # dropless training step: routing + expert-path backward on a route sample
            return time_oracle_train_sample(wn, xn, dy_bits[:n], wr, bias, args.block_m,
                                            n_routes=1024, seed=i, act=act_code(args))
        if args.fp8 or args.mx:
            return time_oracle_sample_fp8(wn, xn, wr, bias, args.block_m, 1, seed_experts=i,
                                          mx=args.mx)
        return time_oracle_sample(wn, xn, wr, bias, args.block_m, max(1, min(4, args.cpu_experts)),
                                  seed_experts=i, act=act_code(args),
                                  prob_in_act=args.prob_in_act)

    # the whole run stays near two minutes of oracle work: a sample that takes
    # longer than its share shrinks the token count of the following ones
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_tok = w.n_tokens

    def run_one(i):
        nonlocal n_tok
        out = sample(i, n_tok)
        if out[2] > budget and n_tok > 64:
            n_tok = max(64, int(n_tok * budget / out[2]) // 64 * 64)
        return out

    for i in range(args.warmup):
        run_one(i)
    vals, secs, descs = [], 0.0, []
    t_start = time.perf_counter()
    for i in range(args.steps):
        n_used = n_tok
        v, desc, s, cores = run_one(i)
        vals.append(v)
        secs += s
        descs.append((n_used, desc))
    desc = descs[-1][1]
    if descs[-1][0] < w.n_tokens:
        desc = ("first %d of the %d tokens as a batch of their own (work per token does not "
                "depend on N): %s" % (descs[-1][0], w.n_tokens, desc))
    wall = time.perf_counter() - t_start
    value = len(vals) / sum(1.0 / v for v in vals)  # tokens over total extrapolated time
    out = {
        "impl": "reference", "metric": METRIC_TRAIN if train else METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        # the host time each timed step actually took (its bounded sample), and
        # the time the oracle would need for the whole step at the same rate
        "ms_per_step": wall / max(1, args.steps) * 1e3,
        "ms_per_step_extrapolated": w.n_tokens / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": w.name, "description": w.note, "block_m": args.block_m,
                                        "parallelism": "single host, OpenMP",
                                        "precision": ("E4M3 GEMM operands, row-wise scales"
                                                      if args.fp8 and not train else
                                                      "MX E4M3 GEMM operands, E8M0 scale per 32 values"
                                                      if args.mx and not train else "bf16 inputs")},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "per step: " + desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(out))
    return 0


# ----------------------------------------------------------------------------- our arm
class GpuCtx:
    """This rank's device and process group."""

    def __init__(self):
        import torch
        self.world, self.rank, self.local = dist_env()
        if not torch.cuda.is_available():
            raise RuntimeError("bench.py needs a CUDA device")
        self.dev = torch.device("cuda", self.local)
        torch.cuda.set_device(self.dev)
        self.dist = init_dist(self.world, "nccl")

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def steps_for(ms_per_step: float, target_ms: float = 1500.0, lo: int = 100, hi: int = 5000) -> int:
    """Steps that make a timed region of about target_ms (long enough for
    several clock samples)."""
    return int(min(hi, max(lo, -(-target_ms // max(ms_per_step, 1e-3)))))


def routing_summary(w, expert_counts, kept_counts, cap):
    """Realised routing of one batch: kept and dropped routes, experts at
    capacity and, for a Zipf workload, route shares against the target by
    popularity rank."""
    import numpy as np
    import synth
    ec = np.asarray(expert_counts, np.int64)
    kc = np.asarray(kept_counts, np.int64)
    R = w.n_tokens * w.top_k
    d = {"routes": R, "kept_routes": int(kc.sum()), "dropped_routes": int(R - kc.sum()),
         "experts_at_capacity": int((ec >= cap).sum()) if cap else 0,
         "experts_without_routes": int((ec == 0).sum())}
    if w.zipf_s is not None:
        ranks = synth.zipf_ranks(w.seed, w.n_experts)
        target = synth.zipf_target_shares(w.n_experts, w.top_k, w.zipf_s)
        share = np.empty(w.n_experts)
        share[ranks - 1] = ec / max(1, R)
        rel = share / target - 1.0
        n64 = min(64, w.n_experts)
        d.update({"zipf_s": w.zipf_s,
                  "share_by_rank_top8": [round(float(v), 5) for v in share[:8]],
                  "target_by_rank_top8": [round(float(v), 5) for v in target[:8]],
                  "ranks_within_10pct_of_target": "%d of ranks 1-%d" % (
                      int((np.abs(rel[:n64]) <= 0.10).sum()), n64),
                  "max_rel_dev_ranks_1_64": float(np.abs(rel[:n64]).max())})
    return d


def run_ours(args):
    ctx = GpuCtx()
    out = forward_bench(args, ctx, args.workload, args.steps, args.warmup, full=True)
    extras = (not args.no_extras and ctx.world == 1 and args.workload == "dsv3" and not args.fp8
              and not args.mx
              and args.activation == "swiglu" and not args.prob_in_act)
    if extras:
        import torch
        torch.cuda.empty_cache()
        q = forward_bench(args, ctx, "qwen3_30b", None, 10, full=False)
        out["qwen3_30b_forward"] = {k: q[k] for k in (
            "value", "unit", "steps", "ms_per_step", "config", "roofline", "grouped_gemm",
            "graph", "kernels_ms", "kernels", "routing", "clocks", "gpu_launches")}
        torch.cuda.empty_cache()
        t = train_bench(args, ctx, "dropless", None, 5, sweep=False, full=False)
        out["dropless_train"] = {k: t[k] for k in (
            "metric", "value", "unit", "steps", "ms_per_step", "config", "roofline",
            "tflops_fwd_bwd", "pct_bf16_peak_fwd_bwd", "calls_ms", "routing", "clocks",
            "gpu_launches")}
        out["extra_lines"] = ("qwen3_30b_forward and dropless_train: the Qwen3-30B-A3B-shaped "
                              "forward and the dropless N=16384 training step, each timed in a "
                              "region of its own (about 1.5 s) with its own clock record")
    if ctx.rank == 0:
        print(json.dumps(out))
    ctx.close()
    return 0


def forward_bench(args, ctx, wname, steps, warmup, full=True):
    """One forward workload timed on this rank. steps None: enough steps for
    about 1.5 s of timed work. full: also the end-to-end leg with host copies
    and the CPU baseline. Returns the JSON object (printed by the caller)."""
    import numpy as np
    import torch

    import mixture_experts_routing_gb300 as moe
    import synth
    import synth.gpu

    world, rank, dev, dist = ctx.world, ctx.rank, ctx.dev, ctx.dist
    w = synth.WORKLOADS[wname]
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    cfg = moe.Config(N, H, E, K, I, w.cap_num, w.cap_den, block_m=args.block_m,
                     activation=act_code(args), prob_in_act=args.prob_in_act)
    peaks = load_peaks()

    # inputs: this rank's batch (seed = rank), shared weights
    rank_seed = w.seed + rank
    x_bits, wr_h, bias_h = host_inputs(w, rank_seed)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    wr = torch.from_numpy(wr_h).to(dev)
    bias = None if bias_h is None else torch.from_numpy(bias_h).to(dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    w13 = torch.empty((E, 2 * I, H), **bf)
    w2 = torch.empty((E, H, I), **bf)
    tmp = torch.empty((E, H, I), **bf)
    synth.gpu.fill(tmp, w.seed, synth.STREAM["wg"], w.w_std)
    wu = torch.empty((E, H, I), **bf)
    synth.gpu.fill(wu, w.seed, synth.STREAM["wu"], w.w_std)
    moe.pack_w13(cfg, tmp, wu, w13)
    del wu
    tmp = tmp.view(E, I, H)
    synth.gpu.fill(tmp, w.seed, synth.STREAM["wd"], w.w_std)
    moe.pack_w2(cfg, tmp, w2)
    torch.cuda.synchronize()
    del tmp
    torch.cuda.empty_cache()
    routes = moe.alloc_routes(cfg, dev)
    ws = moe.alloc_workspace(cfg, dev)
    h, o, y = moe.alloc_buffers(cfg, dev)
    stream = torch.cuda.current_stream(dev)
    mx = args.mx
    fp8 = args.fp8 or mx  # one-byte GEMM operands (row scales, or MX block scales)
    weight_bytes = (w13.numel() + w2.numel()) * (1 if fp8 else 2)
    quant_ms = None
    if fp8:  # weights quantised once, before any step
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        wq = moe.MxWeights(cfg, w13, w2, stream) if mx else moe.Fp8Weights(cfg, w13, w2, stream)
        q1.record(stream)
        torch.cuda.synchronize()
        quant_ms = q0.elapsed_time(q1)
        del w13, w2
        torch.cuda.empty_cache()
        xq, xs, hq, hs = (moe.alloc_mx_buffers if mx else moe.alloc_fp8_buffers)(cfg, dev)

    names = (("route", "quant_x", "fc1", "quant_h", "fc2", "combine") if fp8
             else ("route", "fc1", "fc2", "combine"))

    def step(evs=None, xb=None, yb=None, strm=None):
        xb = x if xb is None else xb
        yb = y if yb is None else yb
        s = stream if strm is None else strm

        def mark(i):
            if evs is not None:
                evs[i].record(s)
        mark(0)
        moe.route_align(cfg, xb, wr, bias, routes, ws, s)
        mark(1)
        if mx:
            moe.quantize_mx_fp8(xb, xq, xs, s)
            mark(2)
            moe.fc1_forward_mx(cfg, routes, xq, xs, wq.w13q, wq.w13_sf, h, s)
            mark(3)
            # only the slots below the padded extent hold routes
            moe.quantize_mx_fp8(h, hq, hs, s, rows_dev=routes.num_tokens_post_padded)
            mark(4)
            moe.fc2_forward_mx(cfg, routes, hq, hs, wq.w2q, wq.w2_sf, o, s)
            mark(5)
        elif fp8:
            moe.quantize_rows_fp8(xb, xq, xs, s)
            mark(2)
            moe.fc1_forward_fp8(cfg, routes, xq, xs, wq.w13q, wq.w13_scale, h, s)
            mark(3)
            # only the slots below the padded extent hold routes
            moe.quantize_rows_fp8(h, hq, hs, s, rows_dev=routes.num_tokens_post_padded)
            mark(4)
            moe.fc2_forward_fp8(cfg, routes, hq, hs, wq.w2q, wq.w2_scale, o, s)
            mark(5)
        else:
            moe.fc1_forward(cfg, routes, xb, w13, h, s)
            mark(2)
            moe.fc2_forward(cfg, routes, h, w2, o, s)
            mark(3)
        moe.combine(cfg, routes, o, yb, s)
        mark(len(names))

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    if steps is None:  # size the timed region from a short untimed probe
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(10):
            step()
        p1.record(stream)
        torch.cuda.synchronize()
        steps = steps_for(p0.elapsed_time(p1) / 10)

    # ---- device-timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index).start()
    time.sleep(0.3)  # let the sampler start before the timed work
    launches0 = moe.launch_count()
    start.record(stream)
    for i in range(steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    launches = moe.launch_count() - launches0
    barrier(dist, dev)
    clk = clocks.stop()
    ms_total = max_over_ranks(start.elapsed_time(end), dist, dev)
    per_kernel = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps))
                  for j, n in enumerate(names)}
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    kept_counts = routes.kept_counts.cpu().numpy()
    expert_counts = routes.expert_counts.cpu().numpy()
    used_slots = int(routes.num_tokens_post_padded.cpu()[0])

    # ---- the whole forward captured as one CUDA graph: 10 warm-up replays,
    # then each replay timed on its own (median and minimum)
    graph = torch.cuda.CUDAGraph()
    gstream = torch.cuda.Stream(dev)
    gstream.wait_stream(stream)
    n0 = moe.launch_count()
    with torch.cuda.graph(graph, stream=gstream):
        step(strm=gstream)
    graph_kernels = moe.launch_count() - n0  # launches recorded into the graph
    stream.wait_stream(gstream)
    for _ in range(10):
        graph.replay()
    reps = max(20, min(steps, 50))
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in gev:
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during the graph replays")
    g_ms = sorted(a.elapsed_time(b) for a, b in gev)
    g_med = statistics.median(g_ms)

    # ---- end to end: every step copies its x in from pinned host memory and
    # its y out to pinned host memory. Two device buffers of each and a copy
    # stream: step i+2's x copy and step i's y copy run under the compute of
    # the steps between (the first two x copies and the last y copies are
    # inside the timed region too).
    ms_e2e = e2e_forward(ctx, stream, step, x, y, x_bits, N, H, steps) if full else None

    model = work_model(w, kept_counts, fp8=fp8, slots=used_slots, mx=mx)
    dom = max(names, key=lambda n: per_kernel[n])
    roof = roofline_for(dom, model, per_kernel[dom], peaks, w.name, fp8=fp8, mx=mx)
    kernels = {n: roofline_for(n, model, per_kernel[n], peaks, w.name, fp8=fp8, mx=mx)
               for n in names}
    gemm_ms = per_kernel["fc1"] + per_kernel["fc2"]
    gemm_flops = model["fc1"]["flops"] + model["fc2"]["flops"]
    issued = 2.0 * 3 * H * I * E * moe.capacity(cfg)
    # the GEMMs' own bound: the weights of the active experts streamed once at
    # the measured HBM rate, or the useful flops at the bf16 peak
    gemm_bound_ms = max((model["fc1"]["bytes"] + model["fc2"]["bytes"]) / (peaks["hbm_gbs"] * 1e9),
                        gemm_flops / (peaks["bf16_tflops"] * (2 if fp8 else 1) * 1e12)) * 1e3

    tokens = N * world * steps
    value = tokens / (ms_total / 1e3)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_total / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "description": w.note, "tokens_per_step_per_gpu": N,
                   "block_m": args.block_m, "capacity": moe.capacity(cfg),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": ("inputs larger than L2 (%.1f GB of expert weights); no flush"
                          % (weight_bytes / 1e9)) if weight_bytes > 129e6 else
                         "expert weights (%.1f MB) fit in L2; no flush" % (weight_bytes / 1e6),
                   **variant_config(args)},
        "gpu_launches": launches,
        "roofline": roof,
        "grouped_gemm": {"ms": gemm_ms, "tflops_useful": gemm_flops / (gemm_ms / 1e3) / 1e12,
                         "pct_bf16_peak": gemm_flops / (gemm_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                         "operands": "e4m3" if fp8 else "bf16",
                         "bound_ms": gemm_bound_ms, "frac_of_bound": gemm_bound_ms / gemm_ms,
                         # the flops a fixed-capacity layer would issue (every slot of
                         # E x cap, empty ones included) over the same time: an
                         # equivalent rate, above the peak when many slots are empty,
                         # since the kernels skip slots past each expert's kept count
                         "tflops_capacity_equivalent": issued / (gemm_ms / 1e3) / 1e12,
                         "capacity_slots_used": model["_kept"] / max(1, E * moe.capacity(cfg)),
                         "kept_routes": model["_kept"], "active_experts": model["_active"]},
        "graph": {"replays": reps, "warmup_replays": 10, "kernels_per_replay": graph_kernels,
                  "median_ms": g_med, "min_ms": g_ms[0],
                  "tokens_per_s_median": N / (g_med / 1e3), "tokens_per_s_min_ms": N / (g_ms[0] / 1e3)},
        "kernels_ms": per_kernel,
        "kernels": {n: {k: v for k, v in kernels[n].items() if k in ("bound", "achieved", "unit", "frac")}
                    for n in names},
        "routing": routing_summary(w, expert_counts, kept_counts, moe.capacity(cfg)),
        "clocks": clk,
    }
    if full:
        out["e2e"] = {"value": N * world * steps / (ms_e2e / 1e3), "unit": UNIT,
                      "h2d_bytes_per_step": N * H * 2, "d2h_bytes_per_step": N * H * 2,
                      "copies": "pinned host x in and y out every step, on a second stream with two "
                                "device buffers each, overlapping the compute of neighbouring steps"}
    if fp8:
        out["config"]["precision"] = (("MX E4M3 GEMM operands with an E8M0 scale per 32 values "
                                       "along the contraction, applied by the tensor cores"
                                       if mx else
                                       "E4M3 GEMM operands with one fp32 scale per row") +
                                      " (w13, w2 once; x and h every step), fp32 accumulation; "
                                      "x, h, o, y in bf16")
        out["weight_quantisation_ms"] = quant_ms
    if full and rank == 0 and world == 1 and not args.no_cpu_baseline:
        if fp8:
            v, desc, secs, cores = time_oracle_sample_fp8(w, x_bits, wr_h, bias_h, args.block_m,
                                                          min(args.cpu_experts, 2), mx=mx)
        else:
            v, desc, secs, cores = time_oracle_sample(w, x_bits, wr_h, bias_h, args.block_m,
                                                      args.cpu_experts, act=act_code(args),
                                                      prob_in_act=args.prob_in_act)
        out["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": desc, "cpu_seconds": secs, "host_cpus": os.cpu_count()}
        if N * H <= 1024 * 512 and not fp8:  # the small layers: also on one thread
            import oracle
            threads = oracle.num_threads()
            oracle.set_num_threads(1)
            try:
                v1, desc1, secs1, _ = time_oracle_sample(w, x_bits, wr_h, bias_h, args.block_m,
                                                         args.cpu_experts, act=act_code(args),
                                                         prob_in_act=args.prob_in_act)
            finally:
                oracle.set_num_threads(threads)
            out["cpu_baseline"]["single_thread"] = {"value": v1, "unit": UNIT, "cores": 1,
                                                    "sample": desc1, "cpu_seconds": secs1}
    return out


def e2e_forward(ctx, stream, step, x, y, x_bits, N, H, steps):
    """Milliseconds (max over ranks) of `steps` forwards, each copying its x in
    from pinned host memory and its y out to pinned host memory."""
    import numpy as np
    import torch
    dev, dist = ctx.dev, ctx.dist
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = [torch.empty((N, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev, y_dev = [x, torch.empty_like(x)], [y, torch.empty_like(y)]
    cstream = torch.cuda.Stream(dev)
    h2d = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(steps, start_evt):
        cstream.wait_event(start_evt)
        with torch.cuda.stream(cstream):
            for b in range(min(2, steps)):
                x_dev[b].copy_(x_host, non_blocking=True)
                h2d[b].record(cstream)
        for i in range(steps):
            b = i % 2
            stream.wait_event(h2d[b])
            step(xb=x_dev[b], yb=y_dev[b])
            done[b].record(stream)
            cstream.wait_event(done[b])
            with torch.cuda.stream(cstream):
                y_host[b].copy_(y_dev[b][:N], non_blocking=True)
                if i + 2 < steps:
                    x_dev[b].copy_(x_host, non_blocking=True)
                h2d[b].record(cstream)
        stream.wait_stream(cstream)

    w0 = torch.cuda.Event()
    w0.record(stream)
    e2e_run(2, w0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_run(steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)
    return max_over_ranks(e0.elapsed_time(e1), dist, dev)


# ----------------------------------------------------------------------------- training step (dropless)
def time_oracle_train_sample(w, x_bits, dy_bits, wr, bias, bm, n_routes=4096, seed=0, act=0):
    """The oracle's routing of every token plus the expert-path backward of a
    bounded sample of routes (forward recompute, dX row, dW contributions),
    extrapolated to all routes by route count."""
    import numpy as np
    import oracle
    import synth
    N, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    t0 = time.perf_counter()
    ids, p, _, _ = oracle.router(x_bits, wr, bias, K, renorm=True)
    t_route = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    r = rng.choice(N * K, size=min(n_routes, N * K), replace=False)
    tok, ex = (r // K).astype(np.int32), ids.ravel()[r].astype(np.int32)
    pr = p.ravel()[r]
    exps = sorted(set(ex.tolist()))
    wg = {e: synth.normal_bf16_bits(w.seed, synth.STREAM["wg"], e * H * I, H * I, w.w_std).reshape(H, I) for e in exps}
    wu = {e: synth.normal_bf16_bits(w.seed, synth.STREAM["wu"], e * H * I, H * I, w.w_std).reshape(H, I) for e in exps}
    wd = {e: synth.normal_bf16_bits(w.seed, synth.STREAM["wd"], e * I * H, I * H, w.w_std).reshape(I, H) for e in exps}
    W = oracle.ExpertWeights(E, wg, wu, wd)
    t0 = time.perf_counter()
    out = oracle.bwd_routes(tok, ex, pr, x_bits, dy_bits, W, H, I, act=act)
    e0 = exps[0]
    sel = ex == e0
    oracle.wgrad_expert(tok[sel], x_bits, dy_bits, out["aw"][sel], out["dg"][sel], out["du"][sel], H, I)
    t_bwd = time.perf_counter() - t0
    t_full = t_route + t_bwd * (N * K) / len(r)
    desc = ("routing of all %d tokens + expert-path backward (recomputed forward, dX, dprob, "
            "dW) of %d of %d routes, time extrapolated by route count" % (N, len(r), N * K))
    return N / t_full, desc, t_route + t_bwd, oracle.num_threads()


def run_ours_train(args):
    ctx = GpuCtx()
    out = train_bench(args, ctx, args.workload, args.steps, args.warmup, sweep=True, full=True)
    if ctx.rank == 0:
        print(json.dumps(out))
    ctx.close()
    return 0


def train_bench(args, ctx, wname, steps, warmup, sweep=True, full=True):
    """Training step of the dropless layer timed on this rank at its full
    token count (and, with sweep, over the N sweep). steps None: enough steps
    for about 1.5 s of timed work. full: also the end-to-end leg with host
    copies and the CPU baseline. Returns the JSON object."""
    import numpy as np
    import torch

    import mixture_experts_routing_gb300 as moe
    import synth
    import synth.gpu

    world, rank, dev, dist = ctx.world, ctx.rank, ctx.dev, ctx.dist
    do_sweep = sweep
    base = synth.WORKLOADS[wname]
    peaks = load_peaks()
    H, E, K, I = base.hidden, base.n_experts, base.top_k, base.inter
    bf = dict(dtype=torch.bfloat16, device=dev)
    # weights, packed once (random-init, the layer's shapes)
    cfg0 = moe.Config(base.n_tokens, H, E, K, I, 0, 1, block_m=args.block_m, ladder=list(base.ladder),
                      ladder_den=base.ladder_den, activation=act_code(args),
                      prob_in_act=args.prob_in_act)
    w13 = torch.empty((E, 2 * I, H), **bf)
    w2 = torch.empty((E, H, I), **bf)
    tmp = torch.empty((E, H, I), **bf)
    synth.gpu.fill(tmp, base.seed, synth.STREAM["wg"], base.w_std)
    wu = torch.empty((E, H, I), **bf)
    synth.gpu.fill(wu, base.seed, synth.STREAM["wu"], base.w_std)
    moe.pack_w13(cfg0, tmp, wu, w13)
    del wu
    tmp = tmp.view(E, I, H)
    synth.gpu.fill(tmp, base.seed, synth.STREAM["wd"], base.w_std)
    moe.pack_w2(cfg0, tmp, w2)
    del tmp
    dw13 = torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev)
    dw2 = torch.empty((E, H, I), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def setup(N):
        w = base.with_tokens(N)
        cfg = moe.Config(N, H, E, K, I, 0, 1, block_m=args.block_m, ladder=list(base.ladder),
                         ladder_den=base.ladder_den, activation=act_code(args),
                         prob_in_act=args.prob_in_act)
        x_bits, wr_h, bias_h = host_inputs(w, w.seed + rank)
        dy_bits = synth.normal_bf16_bits(w.seed + rank, synth.STREAM["dy"], 0, N * H, 1.0).reshape(N, H)
        S = moe.max_slots(cfg)
        st = dict(w=w, cfg=cfg, x_bits=x_bits, dy_bits=dy_bits, wr_h=wr_h, bias_h=bias_h,
                  x=torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(dev),
                  dy=torch.from_numpy(dy_bits.view(np.int16)).view(torch.bfloat16).to(dev),
                  wr=torch.from_numpy(wr_h).to(dev),
                  bias=None if bias_h is None else torch.from_numpy(bias_h).to(dev),
                  routes=moe.alloc_routes(cfg, dev), ws=moe.alloc_workspace(cfg, dev),
                  bws=moe.alloc_backward_workspace(cfg, dev),
                  preact=torch.empty((S, 2 * I), **bf), dx=torch.empty((N, H), **bf),
                  dprob=torch.empty((N, K), dtype=torch.float32, device=dev),
                  rws=moe.alloc_router_backward_workspace(cfg, dev),
                  dwr=torch.empty((H, E), dtype=torch.float32, device=dev),
                  dbias=torch.empty(E, dtype=torch.float32, device=dev))
        st["h"], st["o"], st["y"] = moe.alloc_buffers(cfg, dev)
        st["logits"] = moe.route_workspace_logits(cfg, st["ws"])
        return st

    def step(st, evs=None):
        c, r = st["cfg"], st["routes"]
        if evs is not None:
            evs[0].record(stream)
        moe.route_align(c, st["x"], st["wr"], st["bias"], r, st["ws"], stream)
        if evs is not None:
            evs[1].record(stream)
        moe.ffn_forward_train(c, r, st["x"], w13, w2, st["h"], st["o"], st["preact"], stream)
        if evs is not None:
            evs[2].record(stream)
        moe.combine(c, r, st["o"], st["y"], stream)
        if evs is not None:
            evs[3].record(stream)
        moe.ffn_backward(c, r, st["x"], w13, w2, st["preact"], st["dy"], st["dx"], dw13, dw2,
                         st["dprob"], st["bws"], stream)
        if evs is not None:
            evs[4].record(stream)
        # the logits the forward's route_align left in its workspace
        moe.router_backward(c, r, st["x"], st["wr"], st["bias"], st["dprob"], st["dx"], st["dwr"],
                            st["dbias"], st["rws"], stream, logits=st["logits"])
        if evs is not None:
            evs[5].record(stream)

    def time_steps(st, steps):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist, dev)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(steps):
            step(st, evs[i])
        b.record(stream)
        torch.cuda.synchronize()
        barrier(dist, dev)
        per = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps))
               for j, n in enumerate(("route", "ffn_forward", "combine", "ffn_backward",
                                      "router_backward"))}
        return max_over_ranks(a.elapsed_time(b), dist, dev) / steps, per

    # ---- sweep over N (the curve), then the headline at N = base.n_tokens
    sweep = {}
    for N in (base.sweep if do_sweep else ()):
        if N == base.n_tokens:
            continue
        st = setup(N)
        for _ in range(max(warmup, 3)):
            step(st)
        ms, per = time_steps(st, max(3, min(steps or 10, 10)))
        R = N * K
        sweep[str(N)] = {"ms_per_step": ms, "tokens_per_s": N * world / (ms / 1e3),
                         "tflops": 18.0 * R * H * I / (ms / 1e3) / 1e12,
                         "fwd_ms": per["route"] + per["ffn_forward"] + per["combine"],
                         "bwd_ms": per["ffn_backward"] + per["router_backward"]}
        del st
        torch.cuda.empty_cache()
    st = setup(base.n_tokens)
    N = base.n_tokens
    for _ in range(max(warmup, 3)):
        step(st)
    torch.cuda.synchronize()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    if steps is None:  # size the timed region from a short untimed probe
        probe_ms, _ = time_steps(st, 5)
        steps = steps_for(probe_ms, lo=20, hi=1000)
    clocks = ClockSampler(dev.index).start()
    time.sleep(0.3)
    launches0 = moe.launch_count()
    ms, per = time_steps(st, steps)
    launches = moe.launch_count() - launches0
    clk = clocks.stop()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    R = N * K
    sweep[str(N)] = {"ms_per_step": ms, "tokens_per_s": N * world / (ms / 1e3),
                     "tflops": 18.0 * R * H * I / (ms / 1e3) / 1e12,
                     "fwd_ms": per["route"] + per["ffn_forward"] + per["combine"],
                     "bwd_ms": per["ffn_backward"] + per["router_backward"]}

    # ---- end to end: every step copies x and dY in from pinned host memory
    # and y, dX and dprob out to it. Two sets of these device buffers and a
    # copy stream: a step's copies run under the compute of its neighbours
    # (the first inputs and the last outputs are inside the timed region).
    routing = routing_summary(st["w"], st["routes"].expert_counts.cpu().numpy(),
                              st["routes"].kept_counts.cpu().numpy(), 0)
    ms_e2e = e2e_train(ctx, stream, step, st, N, H, K, steps) if full else None

    bwd_flops = 12.0 * R * H * I
    ach = bwd_flops / (per["ffn_backward"] / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"], "traffic": None, "peak_source": peaks["_source"],
            "kernel": "ffn_backward (FC2 dgrad + SwiGLU backward, FC1 dgrad, dX/dprob "
                      "gather-combine, dW2 and dW13 weight gradients)",
            "ms": per["ffn_backward"], "algorithmic_flops": bwd_flops}
    value = N * world / (ms / 1e3)
    out = {
        "metric": METRIC_TRAIN, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": base.name, "description": base.note, "tokens_per_step_per_gpu": N,
                   "block_m": args.block_m, "ladder": [list(base.ladder), base.ladder_den],
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (%.2f GB of expert weights, %.2f GB of fp32 weight "
                         "gradients); no flush" % ((w13.numel() + w2.numel()) * 2 / 1e9,
                                                   (dw13.numel() + dw2.numel()) * 4 / 1e9),
                   **variant_config(args)},
        "gpu_launches": launches,
        "roofline": roof,
        "tflops_fwd_bwd": 18.0 * R * H * I / (ms / 1e3) / 1e12,
        "pct_bf16_peak_fwd_bwd": 18.0 * R * H * I / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
        "calls_ms": per,
        "routing": routing,
        "clocks": clk,
    }
    if do_sweep:
        out["sweep"] = sweep
    if full:
        out["e2e"] = {"value": N * world / (ms_e2e / 1e3), "unit": UNIT,
                      "h2d_bytes_per_step": 2 * N * H * 2,
                      "d2h_bytes_per_step": 2 * N * H * 2 + N * K * 4,
                      "copies": "pinned host x, dY in and y, dX, dprob out every step, on a "
                                "second stream with two device buffer sets, overlapping "
                                "neighbouring steps"}
    if full and rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, secs, cores = time_oracle_train_sample(st["w"], st["x_bits"], st["dy_bits"],
                                                        st["wr_h"], st["bias_h"], args.block_m,
                                                        act=act_code(args))
        out["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": desc, "cpu_seconds": secs}
    return out


def e2e_train(ctx, stream, step, st, N, H, K, steps):
    """Milliseconds per step (max over ranks) of training steps that each copy
    x and dY in from pinned host memory and y, dX and dprob out to it."""
    import numpy as np
    import torch
    dev, dist = ctx.dev, ctx.dist
    xh = torch.from_numpy(st["x_bits"].view(np.int16)).view(torch.bfloat16).pin_memory()
    dyh = torch.from_numpy(st["dy_bits"].view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = [torch.empty((N, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dxh = [torch.empty((N, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dph = [torch.empty((N, K), dtype=torch.float32).pin_memory() for _ in range(2)]
    io = [st, dict(st, x=torch.empty_like(st["x"]), dy=torch.empty_like(st["dy"]),
                   y=torch.empty_like(st["y"]), dx=torch.empty_like(st["dx"]),
                   dprob=torch.empty_like(st["dprob"]))]
    cstream = torch.cuda.Stream(dev)
    h2d = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(steps, start_evt):
        cstream.wait_event(start_evt)
        with torch.cuda.stream(cstream):
            for b in range(min(2, steps)):
                io[b]["x"].copy_(xh, non_blocking=True)
                io[b]["dy"].copy_(dyh, non_blocking=True)
                h2d[b].record(cstream)
        for i in range(steps):
            b = i % 2
            stream.wait_event(h2d[b])
            step(io[b])
            done[b].record(stream)
            cstream.wait_event(done[b])
            with torch.cuda.stream(cstream):
                yh[b].copy_(io[b]["y"][:N], non_blocking=True)
                dxh[b].copy_(io[b]["dx"], non_blocking=True)
                dph[b].copy_(io[b]["dprob"], non_blocking=True)
                if i + 2 < steps:
                    io[b]["x"].copy_(xh, non_blocking=True)
                    io[b]["dy"].copy_(dyh, non_blocking=True)
                h2d[b].record(cstream)
        stream.wait_stream(cstream)

    w0 = torch.cuda.Event()
    w0.record(stream)
    e2e_run(2, w0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_run(steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)
    return max_over_ranks(e0.elapsed_time(e1), dist, dev) / steps


# ----------------------------------------------------------------------------- serving (graph ladder)
def run_ours_serve(args):
    import numpy as np
    import torch

    import mixture_experts_routing_gb300 as moe
    import synth
    import synth.gpu

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    w = synth.WORKLOADS[args.workload]
    Ntop, H, E, K, I = w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter
    top = moe.Config(Ntop, H, E, K, I, w.cap_num, w.cap_den, block_m=args.block_m,
                     ladder=list(w.ladder), ladder_den=w.ladder_den)
    wr = torch.from_numpy(synth.normal_f32(w.seed, synth.STREAM["wr"], 0, H * E, w.wr_std).reshape(H, E)).to(dev)
    bias = synth.router_bias(w)
    bias = None if bias is None else torch.from_numpy(bias).to(dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    w13, w2 = torch.empty((E, 2 * I, H), **bf), torch.empty((E, H, I), **bf)
    tmp, wu = torch.empty((E, H, I), **bf), torch.empty((E, H, I), **bf)
    synth.gpu.fill(tmp, w.seed, synth.STREAM["wg"], w.w_std)
    synth.gpu.fill(wu, w.seed, synth.STREAM["wu"], w.w_std)
    moe.pack_w13(top, tmp, wu, w13)
    del wu
    tmp = tmp.view(E, I, H)
    synth.gpu.fill(tmp, w.seed, synth.STREAM["wd"], w.w_std)
    moe.pack_w2(top, tmp, w2)
    del tmp
    buckets = sorted({b for b in (128 << i for i in range(16)) if b < Ntop} | {Ntop})
    L = moe.Ladder(top, buckets, args.pad_ratio, wr, bias, w13, w2, dev)
    x_bits = synth.normal_bf16_bits(w.seed + rank, synth.STREAM["x"], 0, Ntop * H, w.x_std).reshape(Ntop, H)
    L.x.copy_(torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(dev))
    # the request sequence: log-uniform batch sizes in [16, Ntop], seeded
    rng = np.random.default_rng(1234 + rank)
    sizes = [int(v) for v in np.exp(rng.uniform(np.log(16), np.log(Ntop), args.serve_batches)).round()]
    stream = torch.cuda.current_stream(dev)
    # eager: the same three calls on exactly n tokens, configs built up front
    cfgs = {n: moe.Config(n, H, E, K, I, w.cap_num, w.cap_den, block_m=args.block_m,
                          ladder=list(w.ladder), ladder_den=w.ladder_den) for n in set(sizes)}

    def eager(n):
        moe.forward(cfgs[n], L.x, wr, bias, w13, w2, L.routes, L.ws, L.h, L.o, L.y, stream)

    def run(fn, reps=1):
        barrier(dist, dev)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record(stream)
        for _ in range(reps):
            for n in sizes:
                fn(n)
        b.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(dist, dev)
        return max_over_ranks(a.elapsed_time(b), dist, dev) / reps, wall / reps

    used = [L.forward(n) for n in sizes]  # warm-up (and the bucket of every batch)
    for _ in range(max(args.warmup - 1, 1)):
        run(L.forward)
    for _ in range(max(args.warmup, 2)):
        run(eager)
    torch.cuda.synchronize()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    reps = max(1, args.steps // 10)
    clocks = ClockSampler(dev.index).start()
    time.sleep(0.3)
    launches0 = moe.launch_count()
    ms_ladder, wall_ladder = run(L.forward, reps)
    launches = (moe.launch_count() - launches0) // reps
    ms_eager, wall_eager = run(eager, reps)
    clk = clocks.stop()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    tokens = sum(sizes) * world

    # end to end through the ladder: each batch's x[:n] comes from pinned host
    # memory and its y[:n] goes back to it. The ladder's graphs are bound to its
    # own x and y buffers, so the host copies go through two staging buffers on
    # a copy stream (batch i+2's x and batch i's y move under the forwards in
    # between) and device copies on the compute stream move the rows in and out.
    xh = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = [torch.empty((Ntop, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    bfd = dict(dtype=torch.bfloat16, device=dev)
    xs = [torch.empty((Ntop, H), **bfd) for _ in range(2)]
    ys = [torch.empty((Ntop, H), **bfd) for _ in range(2)]
    cstream = torch.cuda.Stream(dev)
    h2d = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def e2e_pass(start_evt):
        cstream.wait_event(start_evt)
        with torch.cuda.stream(cstream):
            for b in range(min(2, len(sizes))):
                xs[b][:sizes[b]].copy_(xh[:sizes[b]], non_blocking=True)
                h2d[b].record(cstream)
        for i, n in enumerate(sizes):
            b = i % 2
            stream.wait_event(h2d[b])
            L.x[:n].copy_(xs[b][:n], non_blocking=True)
            L.forward(n)
            ys[b][:n].copy_(L.y[:n], non_blocking=True)
            done[b].record(stream)
            cstream.wait_event(done[b])
            with torch.cuda.stream(cstream):
                yh[b][:n].copy_(ys[b][:n], non_blocking=True)
                if i + 2 < len(sizes):
                    m = sizes[i + 2]
                    xs[b][:m].copy_(xh[:m], non_blocking=True)
                h2d[b].record(cstream)
        stream.wait_stream(cstream)

    w0 = torch.cuda.Event()
    w0.record(stream)
    e2e_pass(w0)
    barrier(dist, dev)
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(reps):
        e2e_pass(ea)
    eb.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)
    ms_e2e = max_over_ranks(ea.elapsed_time(eb), dist, dev) / reps
    out = {
        "metric": METRIC_SERVE, "value": tokens / (ms_ladder / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": reps, "warmup": args.warmup, "ms_per_step": ms_ladder, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "description": w.note, "top_bucket": Ntop, "buckets": buckets,
                   "max_pad_ratio": args.pad_ratio, "batches": len(sizes), "tokens_per_step": sum(sizes),
                   "batch_sizes": sizes, "parallelism": "replicas" if world > 1 else "single GPU",
                   "step": "one pass over the request sequence",
                   "l2": "inputs larger than L2 (%.2f GB of expert weights); no flush"
                         % ((w13.numel() + w2.numel()) * 2 / 1e9)},
        "gpu_launches": launches,
        "e2e": {"value": tokens / (ms_e2e / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": sum(sizes) * H * 2, "d2h_bytes_per_step": sum(sizes) * H * 2,
                "copies": "pinned host x in and y out for every batch through two staging buffers on "
                          "a second stream (overlapping the neighbouring batches), device copies "
                          "into and out of the ladder's buffers"},
        "eager": {"value": tokens / (ms_eager / 1e3), "ms_per_step": ms_eager,
                  "host_wall_ms_per_step": wall_eager * 1e3},
        "ladder_host_wall_ms_per_step": wall_ladder * 1e3,
        "speedup_vs_eager": ms_eager / ms_ladder,
        "replayed_batches": sum(1 for b in used if b >= 0),
        "roofline": None,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(out))
    L.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    import synth
    if args.serve:
        return run_ours_serve(args)
    if synth.WORKLOADS[args.workload].cap_num == 0:
        return run_ours_train(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
