"""Seeded synthetic inputs for the MoE-layer workloads.

This module is shared by the CPU oracle and the CUDA path. It holds no
arithmetic of the MoE layer itself: only the workload shapes, a counter-based
normal generator and the per-expert popularity bias.

Generator definition (``synth_gpu.cu`` implements the same steps on the GPU and
must give the same bits):

1. ``key = mix64((seed << 8) | stream)`` and ``h_i = mix64(key + (i+1)*G)``:
   the i-th output of a SplitMix64 stream (Steele, Lea & Flood, 2014), with
   ``G = 0x9E3779B97F4A7C15`` and ``mix64`` its finaliser.
2. Two uniforms in (0,1), each an odd 24-bit integer times 2^-24 (exact in
   fp32): ``u1`` from bits 41..63 of ``h_i``, ``u2`` from bits 17..39.
3. Box-Muller ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, evaluated with single
   IEEE fp32 operations only (no fused multiply-add). ``ln`` and ``cos`` are
   our own polynomials (atanh series, and Taylor series after exact range
   reduction), so host and device agree bit for bit.
4. ``v = z * std`` in fp32. Tensors stored as bf16 are rounded with
   round-to-nearest-even.

Streams per tensor: x=0, W_r=1, W_gate=2, W_up=3, W_down=4, bias/permutation=5,
dY=6, calibration tokens (used only to fit a stored router bias)=7. Expert weight tensors are indexed in their logical layout
(``W_gate[e,h,i]`` at ``(e*H + h)*I + i``), so any slice can be regenerated
without the rest.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "STREAM", "normal_f32", "normal_bf16_bits",
    "bf16_bits_to_f32", "f32_to_bf16_bits", "zipf_bias", "zipf_ranks", "zipf_target_shares",
    "router_bias", "load_router_bias", "make_host_inputs",
]

STREAM = {"x": 0, "wr": 1, "wg": 2, "wu": 3, "wd": 4, "bias": 5, "dy": 6, "xcal": 7}

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _f(bits: int) -> np.float32:
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


# fp32 constants, given by bit pattern so that both implementations hold the
# same values: sqrt(2), ln 2, 2*pi, 1/(2k+1) for the atanh series,
# (-1)^k/(2k)! for cos and (-1)^k/(2k+1)! for sin.
_SQRT2 = _f(0x3FB504F3)
_LN2 = _f(0x3F317218)
_TWO_PI = _f(0x40C90FDB)
_L9, _L7, _L5, _L3 = _f(0x3DE38E39), _f(0x3E124925), _f(0x3E4CCCCD), _f(0x3EAAAAAB)
_C2, _C4, _C6, _C8, _C10 = (_f(0xBF000000), _f(0x3D2AAAAB), _f(0xBAB60B61),
                            _f(0x37D00D01), _f(0xB493F27E))
_S3, _S5, _S7, _S9 = _f(0xBE2AAAAB), _f(0x3C088889), _f(0xB9500D01), _f(0x3638EF1D)
_ONE = np.float32(1.0)
_HALF = np.float32(0.5)
_QUARTER = np.float32(0.25)
_EIGHTH = np.float32(0.125)
_TWO = np.float32(2.0)
_INV24 = np.float32(2.0 ** -24)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _hash(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        key = _mix64(np.array([(seed << 8) | stream], dtype=np.uint64))[0]
        return _mix64(key + (idx.astype(np.uint64) + np.uint64(1)) * _G)


def _log_f32(u: np.ndarray) -> np.ndarray:
    bits = u.view(np.uint32)
    e = (bits >> np.uint32(23)).astype(np.int32) - 127
    m = ((bits & np.uint32(0x7FFFFF)) | np.uint32(0x3F800000)).view(np.float32)
    big = m > _SQRT2
    m = np.where(big, m * _HALF, m)
    e = e + big.astype(np.int32)
    y = (m - _ONE) / (m + _ONE)
    y2 = y * y
    p = _L9
    p = p * y2 + _L7
    p = p * y2 + _L5
    p = p * y2 + _L3
    p = p * y2 + _ONE
    lnm = (_TWO * y) * p
    return e.astype(np.float32) * _LN2 + lnm


def _cos2pi_f32(u: np.ndarray) -> np.ndarray:
    r = np.where(u < _HALF, u, u - _ONE)
    a = np.abs(r)
    neg = a > _QUARTER
    b = np.where(neg, _HALF - a, a)
    use_sin = b > _EIGHTH
    c = np.where(use_sin, _QUARTER - b, b)
    x = c * _TWO_PI
    x2 = x * x
    pc = _C10
    pc = pc * x2 + _C8
    pc = pc * x2 + _C6
    pc = pc * x2 + _C4
    pc = pc * x2 + _C2
    pc = pc * x2 + _ONE
    ps = _S9
    ps = ps * x2 + _S7
    ps = ps * x2 + _S5
    ps = ps * x2 + _S3
    ps = ps * x2 + _ONE
    ps = ps * x
    v = np.where(use_sin, ps, pc)
    return np.where(neg, -v, v)


_HERE = __import__("os").path.dirname(__import__("os").path.abspath(__file__))
_CLIB = None


def build_host(force: bool = False) -> str:
    """Compile the C twin (synth_host.c) with gcc; returns the library path."""
    import os
    import subprocess
    src = os.path.join(_HERE, "synth_host.c")
    so = os.path.join(_HERE, "libsynth_host.so")
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        tmp = so + ".tmp.%d" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                        "-fPIC", "-shared", src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, so)
    return so


def _clib():
    global _CLIB
    if _CLIB is None:
        import ctypes
        L = ctypes.CDLL(build_host())
        for name in ("synth_normal_f32", "synth_normal_bf16"):
            f = getattr(L, name)
            f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                          ctypes.c_uint32, ctypes.c_float]
            f.restype = None
        _CLIB = L
    return _CLIB


def normal_f32(seed: int, stream: int, start: int, count: int, std: float = 1.0) -> np.ndarray:
    """fp32 values ``z_i * std`` for counter indices ``start .. start+count-1``
    (computed by the C twin; ``normal_f32_numpy`` is the same definition)."""
    out = np.empty(count, dtype=np.float32)
    if count:
        _clib().synth_normal_f32(out.ctypes.data, count, start, seed, stream, float(std))
    return out


def normal_f32_numpy(seed: int, stream: int, start: int, count: int, std: float = 1.0) -> np.ndarray:
    """The generator definition in numpy (slow; pins the C and CUDA twins)."""
    idx = np.arange(start, start + count, dtype=np.uint64)
    out = np.empty(count, dtype=np.float32)
    chunk = 1 << 16
    s32 = np.float32(std)
    for a in range(0, count, chunk):
        h = _hash(seed, stream, idx[a:a + chunk])
        u1 = ((h >> np.uint64(41)).astype(np.uint32) * np.uint32(2) + np.uint32(1)).astype(np.float32) * _INV24
        u2 = (((h >> np.uint64(17)) & np.uint64(0x7FFFFF)).astype(np.uint32) * np.uint32(2)
              + np.uint32(1)).astype(np.float32) * _INV24
        rad = np.sqrt(np.float32(-2.0) * _log_f32(u1))
        out[a:a + chunk] = (rad * _cos2pi_f32(u2)) * s32
    return out


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round-to-nearest-even); inputs are finite."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16_bits(seed: int, stream: int, start: int, count: int, std: float = 1.0) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    if count:
        _clib().synth_normal_bf16(out.ctypes.data, count, start, seed, stream, float(std))
    return out


def zipf_ranks(seed: int, n_experts: int) -> np.ndarray:
    """Popularity rank of each expert (1 = most popular): experts ordered by
    the SplitMix64 output of stream 5 at index e."""
    h = _hash(seed, STREAM["bias"], np.arange(n_experts, dtype=np.uint64))
    order = np.argsort(h, kind="stable")
    rank = np.empty(n_experts, dtype=np.int64)
    rank[order] = np.arange(1, n_experts + 1)
    return rank


def zipf_bias(seed: int, n_experts: int, s: float) -> np.ndarray:
    """Per-expert router bias ``b_e = -s * ln(rank_e)`` (ranks from
    ``zipf_ranks``). Adding ``b`` to the logits scales each expert's softmax
    weight by ``rank^-s``; the route shares that top-K selection then gives
    are steeper than Zipf(s) at the head, so the named workloads use a
    calibrated bias instead (``router_bias``)."""
    rank = zipf_ranks(seed, n_experts)
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


def zipf_target_shares(n_experts: int, top_k: int, s: float) -> np.ndarray:
    """Target route share of each popularity rank (index r-1 for rank r):
    Zipf(s), ``share_r`` proportional to ``r^-s``, summing to 1, with no share
    above 1/K (a token picks an expert at most once, so an expert can hold at
    most N of the N*K routes). Shares over the cap are set to 1/K and the
    others scaled up to keep the sum at 1, repeated until none exceeds it."""
    w = np.arange(1, n_experts + 1, dtype=np.float64) ** (-float(s))
    cap = 1.0 / top_k
    clipped = np.zeros(n_experts, dtype=bool)
    while True:
        free = 1.0 - cap * clipped.sum()
        share = np.where(clipped, cap, w * free / w[~clipped].sum())
        over = (share > cap * (1 + 1e-12)) & ~clipped
        if not over.any():
            return share
        clipped |= over


_BIAS_DIR = __import__("os").path.join(_HERE, "data")


def router_bias_path(name: str) -> str:
    return __import__("os").path.join(_BIAS_DIR, "router_bias_%s.txt" % name)


def load_router_bias(name: str, n_experts: int) -> Optional[np.ndarray]:
    """The stored, calibrated router bias of workload ``name`` (fp32 [E]), or
    None when the workload has none. File format: '#' comments, then one line
    per expert: ``e bits`` with ``bits`` the fp32 bit pattern in hex."""
    import os
    path = router_bias_path(name)
    if not os.path.exists(path):
        return None
    bits = np.zeros(n_experts, dtype=np.uint32)
    seen = np.zeros(n_experts, dtype=bool)
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            e = int(line[0])
            bits[e] = int(line[1], 16)
            seen[e] = True
    if not seen.all():
        raise ValueError("%s: %d of %d experts missing" % (path, int((~seen).sum()), n_experts))
    return bits.view(np.float32).copy()


def router_bias(w: "Workload") -> Optional[np.ndarray]:
    """Router bias of a workload: none for a balanced router; for a Zipf(s)
    workload the stored bias calibrated so that route shares follow Zipf(s)
    (capped at 1/K) when one exists for its name and expert count, else
    ``zipf_bias`` (the small test layers)."""
    if w.zipf_s is None:
        return None
    if w.calibrated_bias:
        b = load_router_bias(w.calibrated_bias, w.n_experts)
        if b is None:
            raise FileNotFoundError(router_bias_path(w.calibrated_bias))
        return b
    return zipf_bias(w.seed, w.n_experts, w.zipf_s)


@dataclass(frozen=True)
class Workload:
    """One MoE-layer forward workload: shapes, capacity factor and input recipe."""
    name: str
    n_tokens: int
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    cap_num: int          # capacity factor F = cap_num / cap_den; 0 means dropless
    cap_den: int
    x_std: float = 1.0
    wr_std: float = 0.02
    w_std: float = 0.02
    zipf_s: Optional[float] = None
    seed: int = 0
    note: str = ""
    sweep: tuple = field(default=())
    ladder: tuple = field(default=())   # dropless: rung multipliers (numerators)
    ladder_den: int = 1
    calibrated_bias: str = ""           # name of the stored calibrated router bias, if any

    def with_tokens(self, n: int) -> "Workload":
        d = dict(self.__dict__)
        d["n_tokens"] = n
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 128, 8, 2, 256, 1, 1,
                     note="tiny MoE layer: N=256, H=128, E=8, top-2, I=256, F=1.0"),
    "qwen3_small": Workload("qwen3_small", 1024, 512, 8, 2, 1024, 5, 4,
                            note="small Qwen3-MoE-style layer: N=1024 (2x512), H=512, E=8, top-2, I=1024, F=1.25"),
    "qwen3_30b": Workload("qwen3_30b", 8192, 2048, 128, 8, 768, 1, 1, zipf_s=1.0,
                          calibrated_bias="qwen3_30b",
                          note="Qwen3-30B-A3B-shaped layer: N=8192, H=2048, E=128, top-8, I=768, F=1.0, Zipf(1.0) router bias"),
    "dsv3": Workload("dsv3", 4096, 7168, 256, 8, 2048, 5, 4, w_std=0.006,
                     note="DeepSeek-V3-shaped layer: N=4096, H=7168, E=256, top-8, I=2048, F=1.25, balanced router"),
    # profiling case: the DeepSeek-V3 shapes with 16 experts and N scaled so that
    # each expert sees the same ~128 routes; 1.4 GB of weights (above L2)
    "dsv3_e16": Workload("dsv3_e16", 256, 7168, 16, 8, 2048, 5, 4, w_std=0.006,
                         note="DeepSeek-V3 shapes with 16 experts, N=256 (ncu profiling case)"),
    # profiling case: the DeepSeek-V3 router shape (N=4096, H=7168, E=256,
    # top-8) with I=128 experts, so the whole problem holds 1.4 GB on the device
    "dsv3_route": Workload("dsv3_route", 4096, 7168, 256, 8, 128, 5, 4, w_std=0.006,
                           note="DeepSeek-V3 router shape with I=128 experts (ncu profiling case)"),
    # profiling case: the dropless per-expert shapes (H=4096, I=1408, ~1536
    # routes per expert) with 16 experts and N=4096, about 3 GB on the device
    "dropless_e16": Workload("dropless_e16", 4096, 4096, 16, 6, 1408, 0, 1, zipf_s=0.8,
                             note="dropless per-expert shapes with 16 experts, N=4096 (ncu profiling case)",
                             ladder=(2, 3, 4, 5, 6, 8), ladder_den=4, calibrated_bias="dropless_e16"),
    "dropless": Workload("dropless", 16384, 4096, 64, 6, 1408, 0, 1, zipf_s=0.8,
                         note="dropless bucketed layer: H=4096, E=64, top-6, I=1408, N swept 128..16384, Zipf(0.8)",
                         sweep=tuple(2 ** k for k in range(7, 15)),
                         ladder=(2, 3, 4, 5, 6, 8), ladder_den=4, calibrated_bias="dropless"),
}


def make_host_inputs(w: Workload, experts: Optional[list] = None) -> dict:
    """Host copies of a workload's inputs (bf16 as uint16 bit patterns).

    ``experts`` restricts the expert weights to a subset (returned as dicts
    keyed by expert id); None generates all of them.
    """
    N, H, E, I = w.n_tokens, w.hidden, w.n_experts, w.inter
    out = {
        "x": normal_bf16_bits(w.seed, STREAM["x"], 0, N * H, w.x_std).reshape(N, H),
        "wr": normal_f32(w.seed, STREAM["wr"], 0, H * E, w.wr_std).reshape(H, E),
        "bias": router_bias(w),
    }
    ids = range(E) if experts is None else experts
    for name in ("wg", "wu"):
        out[name] = {e: normal_bf16_bits(w.seed, STREAM[name], e * H * I, H * I, w.w_std).reshape(H, I)
                     for e in ids}
    out["wd"] = {e: normal_bf16_bits(w.seed, STREAM["wd"], e * I * H, I * H, w.w_std).reshape(I, H)
                 for e in ids}
    return out
