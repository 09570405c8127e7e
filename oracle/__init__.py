"""CPU oracle of the capacity-bounded MoE layer forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``. The library never imports it, and it
imports nothing from the library.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp32, fixed evaluation
order; see its header for the steps and the passages they follow). This module
compiles it with gcc and wraps it with ctypes; the only Python-side logic is
array marshalling and the slot layout bookkeeping of ``route()``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to the source (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
               "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        L.oracle_exp.argtypes = [f32]
        L.oracle_exp.restype = f32
        L.oracle_capacity.argtypes = [i64, i64, i64, i64, i64]
        L.oracle_capacity.restype = i64
        L.oracle_router.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
        L.oracle_router.restype = i32
        L.oracle_select_layout.argtypes = [i32, i32, i32, i64, i32, P, P, P, P, P, P, P, P, P, P]
        L.oracle_select_layout.restype = i32
        L.oracle_ffn_routes.argtypes = [i32, P, P, i32, i32, P, P, P, P, i32, P, P, P]
        L.oracle_ffn_routes.restype = i32
        L.oracle_combine.argtypes = [i32, i32, i32, i32, P, P, P, P]
        L.oracle_combine.restype = i32
        L.oracle_forward_tokens.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i32, i32,
                                            P]
        L.oracle_forward_tokens.restype = i32
        L.oracle_num_threads.restype = i32
        L.oracle_set_num_threads.argtypes = [i32]
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def exp_f32(v: np.ndarray) -> np.ndarray:
    L = lib()
    v = np.asarray(v, dtype=np.float32).ravel()
    return np.array([L.oracle_exp(float(a)) for a in v], dtype=np.float32)


def capacity(N: int, K: int, E: int, cap_num: int, cap_den: int) -> int:
    return int(lib().oracle_capacity(N, K, E, cap_num, cap_den))


def router(x_bits: np.ndarray, wr: np.ndarray, bias: Optional[np.ndarray], K: int,
           renorm: bool = True, want_probs: bool = False, want_logits: bool = False):
    """Returns (topk_ids [N,K] i32, topk_p [N,K] f32, probs [N,E] or None, logits or None)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    N, H = x_bits.shape
    E = wr.shape[1]
    ids = np.empty((N, K), dtype=np.int32)
    p = np.empty((N, K), dtype=np.float32)
    probs = np.empty((N, E), dtype=np.float32) if want_probs else None
    logits = np.empty((N, E), dtype=np.float32) if want_logits else None
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rc = lib().oracle_router(N, H, E, K, int(bool(renorm)), _p(x_bits), _p(wr), _p(b), _p(ids),
                             _p(p), _p(probs), _p(logits))
    if rc != 0:
        raise RuntimeError("oracle_router failed: %d" % rc)
    return ids, p, probs, logits


@dataclass
class Layout:
    cap: int
    cpad: int
    keep: np.ndarray             # [N,K] u8
    expert_counts: np.ndarray    # [E]
    kept_counts: np.ndarray      # [E]
    sorted_slot_ids: np.ndarray  # [E*cpad]
    expert_ids: np.ndarray       # [E*cpad/bm]
    block_start: np.ndarray      # [E]
    num_tokens_post_padded: int
    token_routes: np.ndarray     # [N,K]


def select_layout(topk_ids: np.ndarray, topk_p: np.ndarray, E: int, cap: int, bm: int) -> Layout:
    topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    topk_p = np.ascontiguousarray(topk_p, dtype=np.float32)
    N, K = topk_ids.shape
    cpad = (cap + bm - 1) // bm * bm
    keep = np.empty((N, K), dtype=np.uint8)
    ec = np.empty(E, dtype=np.int32)
    kc = np.empty(E, dtype=np.int32)
    ssi = np.empty(max(E * cpad, 1), dtype=np.int32)
    eid = np.empty(max(E * cpad // bm, 1), dtype=np.int32)
    bs = np.empty(E, dtype=np.int32)
    ntpp = np.zeros(1, dtype=np.int32)
    tr = np.empty((N, K), dtype=np.int32)
    rc = lib().oracle_select_layout(N, E, K, cap, bm, _p(topk_ids), _p(topk_p), _p(keep), _p(ec),
                                    _p(kc), _p(ssi), _p(eid), _p(bs), _p(ntpp), _p(tr))
    if rc != 0:
        raise RuntimeError("oracle_select_layout failed: %d" % rc)
    return Layout(cap, cpad, keep, ec, kc, ssi[:E * cpad], eid[:E * cpad // bm], bs,
                  int(ntpp[0]), tr)


class ExpertWeights:
    """Per-expert bf16 weight blocks held as pointer tables for the C side.

    wg[e], wu[e]: [H,I] bit patterns; wd[e]: [I,H]. Experts not present are
    null pointers (using one is a caller error)."""

    def __init__(self, E: int, wg: Dict[int, np.ndarray], wu: Dict[int, np.ndarray],
                 wd: Dict[int, np.ndarray]):
        self._keep = []
        PT = ctypes.c_void_p * E
        self.wg, self.wu, self.wd = PT(), PT(), PT()
        for table, src in ((self.wg, wg), (self.wu, wu), (self.wd, wd)):
            for e, a in src.items():
                a = np.ascontiguousarray(a, dtype=np.uint16)
                self._keep.append(a)
                table[e] = a.ctypes.data


ACT_SILU, ACT_GELU = 0, 1


def ffn_routes(tokens: Sequence[int], experts: Sequence[int], x_bits: np.ndarray,
               W: ExpertWeights, H: int, I: int, want_h: bool = False, act: int = ACT_SILU,
               scales: Optional[np.ndarray] = None):
    """FFN output o [n,H] (and activation a [n,I]) of the given (token, expert)
    pairs; act: 0 silu, 1 gelu; scales [n]: per-route factor of the activation
    (p' when the routing probability is applied in the activation)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    n = len(tokens)
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    o = np.empty((n, H), dtype=np.float32)
    h = np.empty((n, I), dtype=np.float32) if want_h else None
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    rc = lib().oracle_ffn_routes(n, _p(tokens), _p(experts), H, I, _p(x_bits), W.wg, W.wu, W.wd,
                                 int(act), _p(sc), _p(h), _p(o))
    if rc != 0:
        raise RuntimeError("oracle_ffn_routes failed: %d" % rc)
    return (o, h) if want_h else o


def combine(t0: int, t1: int, keep: np.ndarray, topk_p: Optional[np.ndarray],
            o_routes: np.ndarray) -> np.ndarray:
    """topk_p None: unit weights."""
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    topk_p = None if topk_p is None else np.ascontiguousarray(topk_p, dtype=np.float32)
    o_routes = np.ascontiguousarray(o_routes, dtype=np.float32)
    K = keep.shape[1]
    H = o_routes.shape[-1]
    y = np.empty((t1 - t0, H), dtype=np.float32)
    lib().oracle_combine(t0, t1, K, H, _p(keep), _p(topk_p), _p(o_routes), _p(y))
    return y


def forward_tokens(t0: int, t1: int, x_bits: np.ndarray, W: ExpertWeights, H: int, I: int,
                   topk_ids: np.ndarray, topk_p: np.ndarray, keep: np.ndarray, act: int = ACT_SILU,
                   prob_in_act: bool = False) -> np.ndarray:
    """Layer output y [t1-t0, H] (fp32) for tokens [t0, t1); act 0 silu, 1 gelu;
    prob_in_act: p' multiplies the activation and the combine uses unit weights."""
    K = topk_ids.shape[1]
    y = np.empty((max(t1 - t0, 0), H), dtype=np.float32)
    rc = lib().oracle_forward_tokens(t0, t1, K, H, I, _p(np.ascontiguousarray(x_bits, dtype=np.uint16)),
                                     W.wg, W.wu, W.wd,
                                     _p(np.ascontiguousarray(topk_ids, dtype=np.int32)),
                                     _p(np.ascontiguousarray(topk_p, dtype=np.float32)),
                                     _p(np.ascontiguousarray(keep, dtype=np.uint8)), int(act),
                                     int(bool(prob_in_act)), _p(y))
    if rc != 0:
        raise RuntimeError("oracle_forward_tokens failed: %d" % rc)
    return y


@dataclass
class Routing:
    topk_ids: np.ndarray
    topk_p: np.ndarray
    layout: Layout


def route(x_bits: np.ndarray, wr: np.ndarray, bias: Optional[np.ndarray], E: int, K: int,
          cap_num: int, cap_den: int, bm: int, renorm: bool = True) -> Routing:
    """Steps 1-4: router, capacity, selection and layout for all tokens."""
    N = x_bits.shape[0]
    ids, p, _, _ = router(x_bits, wr, bias, K, renorm)
    cap = capacity(N, K, E, cap_num, cap_den)
    return Routing(ids, p, select_layout(ids, p, E, cap, bm))


# ---------------------------------------------------------------- dropless variant + backward
def _bind_backward(L):
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    if getattr(L, "_bwd_bound", False):
        return L
    L.oracle_dropless_extent.argtypes = [i64, i64, i64, i32, P, i32, i32]
    L.oracle_dropless_extent.restype = i64
    L.oracle_dropless_layout.argtypes = [i32, i32, i32, i32, P, i32, i32, i64, P, P, P, P, P, P, P,
                                         P]
    L.oracle_dropless_layout.restype = i32
    L.oracle_bwd_routes.argtypes = [i32, P, P, P, i32, i32, i32, P, P, P, P, P, P, P, P, P, P]
    L.oracle_bwd_routes.restype = i32
    L.oracle_wgrad_expert.argtypes = [i32, P, i32, i32, P, P, P, P, P, P, P, P]
    L.oracle_wgrad_expert.restype = i32
    L.oracle_router_backward.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
    L.oracle_router_backward.restype = i32
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_decode.restype = ctypes.c_float
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_quantize_rows_fp8.argtypes = [i32, i32, P, P, P]
    L.oracle_quantize_rows_fp8.restype = i32
    L.oracle_fc1_fp8_routes.argtypes = [i32, P, P, i32, i32, P, P, P, P, i32, P, P]
    L.oracle_fc1_fp8_routes.restype = i32
    L.oracle_fc2_fp8_routes.argtypes = [i32, P, i32, i32, P, P, P, P, P]
    L.oracle_fc2_fp8_routes.restype = i32
    L.oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e8m0_decode.restype = ctypes.c_float
    L.oracle_quantize_mx_fp8.argtypes = [i32, i32, P, P, P]
    L.oracle_quantize_mx_fp8.restype = i32
    L.oracle_fc1_mx_routes.argtypes = [i32, P, P, i32, i32, P, P, P, P, i32, P, P]
    L.oracle_fc1_mx_routes.restype = i32
    L.oracle_fc2_mx_routes.argtypes = [i32, P, i32, i32, P, P, P, P, P]
    L.oracle_fc2_mx_routes.restype = i32
    L._bwd_bound = True
    return L


def dropless_extent(count: int, R: int, E: int, bm: int, ladder_num, ladder_den: int) -> int:
    L = _bind_backward(lib())
    lad = np.ascontiguousarray(ladder_num, dtype=np.int32)
    return int(L.oracle_dropless_extent(count, R, E, bm, _p(lad), len(lad), ladder_den))


def dropless_s_max(N: int, K: int, E: int, bm: int, ladder_num, ladder_den: int) -> int:
    """Static slot bound: R + E * (top rung + bm)."""
    R = N * K
    top = dropless_extent(0, R, E, bm, [max(ladder_num)], ladder_den) if len(ladder_num) else 0
    return R + E * (top + bm)


@dataclass
class DroplessLayout:
    expert_counts: np.ndarray
    extents: np.ndarray
    block_start: np.ndarray
    sorted_slot_ids: np.ndarray   # [s_max]
    expert_ids: np.ndarray        # [s_max / bm]
    num_tokens_post_padded: int
    token_routes: np.ndarray      # [N, K]


def dropless_layout(topk_ids: np.ndarray, E: int, bm: int, ladder_num, ladder_den: int) -> DroplessLayout:
    L = _bind_backward(lib())
    topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    N, K = topk_ids.shape
    lad = np.ascontiguousarray(ladder_num, dtype=np.int32)
    s_max = dropless_s_max(N, K, E, bm, lad, ladder_den)
    ec, ex, bs = (np.empty(E, np.int32) for _ in range(3))
    ssi = np.empty(s_max, np.int32)
    eid = np.empty(s_max // bm, np.int32)
    ntpp = np.zeros(1, np.int32)
    tr = np.empty((N, K), np.int32)
    rc = L.oracle_dropless_layout(N, E, K, bm, _p(lad), len(lad), ladder_den, s_max, _p(topk_ids),
                                  _p(ec), _p(ex), _p(bs), _p(ssi), _p(eid), _p(ntpp), _p(tr))
    if rc != 0:
        raise RuntimeError("oracle_dropless_layout failed: %d" % rc)
    return DroplessLayout(ec, ex, bs, ssi, eid, int(ntpp[0]), tr)


def bwd_routes(tokens, experts, probs, x_bits, dy_bits, W: ExpertWeights, H: int, I: int,
               act: int = ACT_SILU):
    """Per-route backward: (dprob [n], dxr [n,H], dg [n,I], du [n,I], aw [n,I])."""
    L = _bind_backward(lib())
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    probs = np.ascontiguousarray(probs, dtype=np.float32)
    n = len(tokens)
    out = dict(dprob=np.empty(n, np.float32), dxr=np.empty((n, H), np.float32),
               dg=np.empty((n, I), np.float32), du=np.empty((n, I), np.float32),
               aw=np.empty((n, I), np.float32))
    rc = L.oracle_bwd_routes(n, _p(tokens), _p(experts), _p(probs), H, I, int(act),
                             _p(np.ascontiguousarray(x_bits, dtype=np.uint16)),
                             _p(np.ascontiguousarray(dy_bits, dtype=np.uint16)), W.wg, W.wu, W.wd,
                             _p(out["dprob"]), _p(out["dxr"]), _p(out["dg"]), _p(out["du"]),
                             _p(out["aw"]))
    if rc != 0:
        raise RuntimeError("oracle_bwd_routes failed: %d" % rc)
    return out


def wgrad_expert(tokens, x_bits, dy_bits, aw, dg, du, H: int, I: int):
    """(dWd [I,H], dWg [H,I], dWu [H,I]) of one expert from its routes in slot order."""
    L = _bind_backward(lib())
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = len(tokens)
    dwd = np.empty((I, H), np.float32)
    dwg = np.empty((H, I), np.float32)
    dwu = np.empty((H, I), np.float32)
    L.oracle_wgrad_expert(n, _p(tokens), H, I, _p(np.ascontiguousarray(x_bits, dtype=np.uint16)),
                          _p(np.ascontiguousarray(dy_bits, dtype=np.uint16)),
                          _p(np.ascontiguousarray(aw, dtype=np.float32)),
                          _p(np.ascontiguousarray(dg, dtype=np.float32)),
                          _p(np.ascontiguousarray(du, dtype=np.float32)), _p(dwd), _p(dwg), _p(dwu))
    return dwd, dwg, dwu


def backward_all(x_bits, dy_bits, W: ExpertWeights, H: int, I: int, E: int, topk_ids, topk_p,
                 token_routes, act: int = ACT_SILU):
    """Whole expert-path backward: dX [N,H], dprob [N,K], dW per expert (dicts).
    Routes are processed in slot order per expert (token_routes gives the slot)."""
    N, K = topk_ids.shape
    r = np.nonzero(token_routes.ravel() >= 0)[0]
    tok, kk = r // K, r % K
    ex = topk_ids.ravel()[r]
    pr = topk_p.ravel()[r]
    out = bwd_routes(tok, ex, pr, x_bits, dy_bits, W, H, I, act=act)
    dX = np.zeros((N, H), np.float32)
    for k in range(K):  # k order
        m = kk == k
        dX[tok[m]] = dX[tok[m]] + out["dxr"][m]
    dprob = np.zeros((N, K), np.float32)
    dprob[tok, kk] = out["dprob"]
    slots = token_routes.ravel()[r]
    dW = {}
    for e in range(E):
        sel = np.nonzero(ex == e)[0]
        sel = sel[np.argsort(slots[sel], kind="stable")]
        dW[e] = wgrad_expert(tok[sel], x_bits, dy_bits, out["aw"][sel], out["dg"][sel],
                             out["du"][sel], H, I)
    return dX, dprob, dW


def router_backward(x_bits, wr, bias, K: int, dprob, renorm: bool = True, want_dx: bool = True,
                    want_dwr: bool = True):
    """Router backward for a given dprob [N,K] (d loss / d p'): the forward
    router (probabilities and chosen experts) is recomputed by the oracle.
    Returns dict(dlogits [N,E], dwr [H,E], dbias [E], dx [N,H] (router path),
    topk_ids, probs)."""
    L = _bind_backward(lib())
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    N, H = x_bits.shape
    E = wr.shape[1]
    ids, _, probs, _ = router(x_bits, wr, bias, K, renorm=renorm, want_probs=True)
    dprob = np.ascontiguousarray(dprob, dtype=np.float32)
    out = dict(dlogits=np.empty((N, E), np.float32), dbias=np.empty(E, np.float32),
               dwr=np.empty((H, E), np.float32) if want_dwr else None,
               dx=np.empty((N, H), np.float32) if want_dx else None, topk_ids=ids, probs=probs)
    rc = L.oracle_router_backward(N, H, E, K, int(bool(renorm)), _p(x_bits), _p(wr), _p(probs),
                                  _p(ids), _p(dprob), _p(out["dlogits"]), _p(out["dwr"]),
                                  _p(out["dbias"]), _p(out["dx"]))
    if rc != 0:
        raise RuntimeError("oracle_router_backward failed: %d" % rc)
    return out


# ---------------------------------------------------------------- FP8 (E4M3)
def e4m3_decode(codes) -> np.ndarray:
    L = _bind_backward(lib())
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.oracle_e4m3_decode(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    L = _bind_backward(lib())
    v = np.asarray(values, dtype=np.float32)
    return np.array([L.oracle_e4m3_encode(float(a)) for a in v.ravel()], np.uint8).reshape(v.shape)


def quantize_rows_fp8(m_bits: np.ndarray):
    """Row-wise E4M3 quantisation of a bf16 matrix: (codes [rows, cols] u8, scales [rows] f32)."""
    L = _bind_backward(lib())
    m = np.ascontiguousarray(m_bits, dtype=np.uint16)
    rows, cols = m.shape
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty(rows, np.float32)
    L.oracle_quantize_rows_fp8(rows, cols, _p(m), _p(q), _p(sc))
    return q, sc


def fc1_fp8_routes(tokens, experts, xq, xs, wq13, ws13, H: int, I: int, act: int = ACT_SILU,
                   scales=None) -> np.ndarray:
    """h [n, I] of FC1 in FP8 for (token, expert) routes; wq13 [E,2I,H] u8, ws13 [E,2I] f32."""
    L = _bind_backward(lib())
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    n = len(tokens)
    h = np.empty((n, I), np.float32)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    L.oracle_fc1_fp8_routes(n, _p(tokens), _p(experts), H, I, _p(np.ascontiguousarray(xq, np.uint8)),
                            _p(np.ascontiguousarray(xs, np.float32)),
                            _p(np.ascontiguousarray(wq13, np.uint8)),
                            _p(np.ascontiguousarray(ws13, np.float32)), int(act), _p(sc), _p(h))
    return h


def fc2_fp8_routes(experts, hq, hs, wq2, ws2, H: int, I: int) -> np.ndarray:
    """o [n, H] of FC2 in FP8 for routes of the given experts; hq [n, I] u8 and
    hs [n] f32 the routes' quantised h rows, wq2 [E,H,I] u8, ws2 [E,H] f32."""
    L = _bind_backward(lib())
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    n = len(experts)
    o = np.empty((n, H), np.float32)
    L.oracle_fc2_fp8_routes(n, _p(experts), H, I, _p(np.ascontiguousarray(hq, np.uint8)),
                            _p(np.ascontiguousarray(hs, np.float32)),
                            _p(np.ascontiguousarray(wq2, np.uint8)),
                            _p(np.ascontiguousarray(ws2, np.float32)), _p(o))
    return o


# ---------------------------------------------------------------- MX block-scaled FP8
def e8m0_decode(codes) -> np.ndarray:
    L = _bind_backward(lib())
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.oracle_e8m0_decode(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def quantize_mx_fp8(m_bits: np.ndarray):
    """MX quantisation of a bf16 matrix along its rows in blocks of 32:
    (E4M3 codes [rows, cols] u8, E8M0 scale codes [rows, cols/32] u8)."""
    L = _bind_backward(lib())
    m = np.ascontiguousarray(m_bits, dtype=np.uint16)
    rows, cols = m.shape
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty((rows, cols // 32), np.uint8)
    if L.oracle_quantize_mx_fp8(rows, cols, _p(m), _p(q), _p(sc)) != 0:
        raise ValueError("columns must be a multiple of 32")
    return q, sc


def fc1_mx_routes(tokens, experts, xq, xs, wq13, ws13, H: int, I: int, act: int = ACT_SILU,
                  scales=None) -> np.ndarray:
    """h [n, I] of FC1 on MX operands; xq [N,H] u8, xs [N,H/32] u8 (E8M0),
    wq13 [E,2I,H] u8, ws13 [E*2I, H/32] u8."""
    L = _bind_backward(lib())
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    n = len(tokens)
    h = np.empty((n, I), np.float32)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    rc = L.oracle_fc1_mx_routes(n, _p(tokens), _p(experts), H, I, _p(np.ascontiguousarray(xq, np.uint8)),
                                _p(np.ascontiguousarray(xs, np.uint8)),
                                _p(np.ascontiguousarray(wq13, np.uint8)),
                                _p(np.ascontiguousarray(ws13, np.uint8)), int(act), _p(sc), _p(h))
    if rc != 0:
        raise ValueError("H must be a multiple of 32")
    return h


def fc2_mx_routes(experts, hq, hs, wq2, ws2, H: int, I: int) -> np.ndarray:
    """o [n, H] of FC2 on MX operands; hq [n, I] u8 and hs [n, I/32] u8 the
    routes' quantised h rows, wq2 [E,H,I] u8, ws2 [E*H, I/32] u8."""
    L = _bind_backward(lib())
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    n = len(experts)
    o = np.empty((n, H), np.float32)
    rc = L.oracle_fc2_mx_routes(n, _p(experts), H, I, _p(np.ascontiguousarray(hq, np.uint8)),
                                _p(np.ascontiguousarray(hs, np.uint8)),
                                _p(np.ascontiguousarray(wq2, np.uint8)),
                                _p(np.ascontiguousarray(ws2, np.uint8)), _p(o))
    if rc != 0:
        raise ValueError("I must be a multiple of 32")
    return o
