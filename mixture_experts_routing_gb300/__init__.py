"""Capacity-bounded Mixture-of-Experts layer forward for NVIDIA GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/moe.h`` (``libmoe.so``,
built in-tree by ``_build.build()``). The binding only marshals arguments:
every step of the layer runs in the library's CUDA kernels. PyTorch is used
for device memory and streams. If the library is missing, every call raises;
there is no fallback path.

Typical use (all tensors on one CUDA device)::

    cfg = Config(n_tokens=N, hidden=H, n_experts=E, top_k=K, inter=I,
                 cap_num=5, cap_den=4, block_m=32)
    routes = alloc_routes(cfg, device)
    ws = alloc_workspace(cfg, device)
    pack_w13(cfg, w_gate, w_up, w13); pack_w2(cfg, w_down, w2)   # once
    route_align(cfg, x, w_router, bias, routes, ws)
    ffn_forward(cfg, routes, x, w13, w2, h, o)
    combine(cfg, routes, o, y)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "Config", "Routes", "ACT_SWIGLU", "ACT_GEGLU", "MoEError", "lib", "library_path", "alloc_routes", "alloc_workspace",
    "alloc_buffers", "capacity", "max_slots", "max_blocks", "route_workspace_bytes",
    "route_align", "fc1_forward", "fc2_forward", "ffn_forward", "combine", "pack_w13",
    "pack_w2", "status_string", "launch_count", "device_error", "forward",
    "ffn_forward_train", "backward_workspace_bytes", "alloc_backward_workspace", "ffn_backward",
    "router_backward_workspace_bytes", "alloc_router_backward_workspace", "router_backward",
    "Ladder", "ladder_pick",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libmoe.so")
_lib = None

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__("%s failed: %d (%s)" % (fn, status, status_string(status)))
        self.status = status


ACT_SWIGLU, ACT_GEGLU = 0, 1


class Config(ctypes.Structure):
    """Mirror of moe_config_t."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_tokens", "hidden", "n_experts", "top_k", "inter", "cap_num", "cap_den", "block_m",
        "renorm", "ladder_len", "ladder_den")] + [("ladder_num", ctypes.POINTER(ctypes.c_int32)),
                                                  ("activation", ctypes.c_int32),
                                                  ("prob_in_act", ctypes.c_int32),
                                                  ("n_valid", ctypes.c_void_p)]

    def __init__(self, n_tokens, hidden, n_experts, top_k, inter, cap_num=1, cap_den=1,
                 block_m=32, renorm=1, ladder=None, ladder_den=1, activation=ACT_SWIGLU,
                 prob_in_act=0):
        """cap_num=0 selects the dropless layout; ladder: rung multipliers
        (numerators over ladder_den) of the expected rows per expert;
        activation: ACT_SWIGLU or ACT_GEGLU; prob_in_act: p' multiplies the
        activation (unit-weight combine) instead of weighting the combine."""
        lad = list(ladder or [])
        self._ladder = (ctypes.c_int32 * max(len(lad), 1))(*lad)
        super().__init__(n_tokens, hidden, n_experts, top_k, inter, cap_num, cap_den, block_m,
                         renorm, len(lad), ladder_den,
                         ctypes.cast(self._ladder, ctypes.POINTER(ctypes.c_int32)), activation,
                         int(bool(prob_in_act)), None)


class _RoutesC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "topk_ids", "topk_p", "keep", "expert_counts", "kept_counts", "sorted_slot_ids",
        "expert_ids", "block_start", "num_tokens_post_padded", "token_routes", "gemm_sched",
        "slot_prob")]


class _LayerBufsC(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("w_router", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("routes", _RoutesC),
                ("route_workspace", ctypes.c_void_p), ("route_workspace_bytes", ctypes.c_size_t),
                ("h", ctypes.c_void_p), ("o", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("n_valid", ctypes.c_void_p)]


class Routes:
    """Routing metadata tensors (device), allocated to the static bounds."""
    FIELDS = _RoutesC._fields_

    def __init__(self, **tensors):
        for name, _ in self.FIELDS:
            setattr(self, name, tensors[name])

    def c(self) -> _RoutesC:
        return _RoutesC(*[getattr(self, n).data_ptr() for n, _ in self.FIELDS])


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libmoe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libmoe.so is not built (run __graft_entry__.build() or "
                               "python -m mixture_experts_routing_gb300._build)")
        L = ctypes.CDLL(_LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        CP = ctypes.POINTER(Config)
        RP = ctypes.POINTER(_RoutesC)
        for name in ("moe_capacity", "moe_max_slots", "moe_max_blocks", "moe_route_workspace_bytes",
                     "moe_backward_workspace_bytes", "moe_router_backward_workspace_bytes"):
            getattr(L, name).argtypes = [CP]
            getattr(L, name).restype = I64
        L.moe_route_align.argtypes = [CP, P, P, P, RP, P, SZ, P]
        L.moe_fc1_forward.argtypes = [CP, RP, P, P, P, P]
        L.moe_fc2_forward.argtypes = [CP, RP, P, P, P, P]
        L.moe_ffn_forward.argtypes = [CP, RP, P, P, P, P, P, P]
        L.moe_combine.argtypes = [CP, RP, P, P, P]
        L.moe_ffn_forward_train.argtypes = [CP, RP, P, P, P, P, P, P, P]
        L.moe_ffn_backward.argtypes = [CP, RP, P, P, P, P, P, P, P, P, P, P, SZ, P]
        L.moe_router_backward.argtypes = [CP, RP, P, P, P, P, P, P, P, P, P, SZ, P]
        L.moe_route_workspace_logits.argtypes = [CP, P]
        L.moe_route_workspace_logits.restype = P
        L.moe_ladder_pick.argtypes = [P, I32, ctypes.c_int32, ctypes.c_float]
        L.moe_ladder_pick.restype = I32
        L.moe_ladder_create.argtypes = [CP, P, I32, ctypes.c_float, ctypes.POINTER(_LayerBufsC),
                                        ctypes.POINTER(ctypes.c_void_p)]
        L.moe_ladder_forward.argtypes = [P, ctypes.c_int32, P, ctypes.POINTER(ctypes.c_int)]
        L.moe_ladder_destroy.argtypes = [P]
        for name in ("moe_ladder_create", "moe_ladder_forward", "moe_ladder_destroy"):
            getattr(L, name).restype = I32
        L.moe_pack_w13.argtypes = [CP, P, P, P, P]
        L.moe_pack_w2.argtypes = [CP, P, P, P]
        L.moe_quantize_rows_fp8.argtypes = [P, I64, P, I32, P, P, P]
        L.moe_fc1_forward_fp8.argtypes = [CP, RP, P, P, P, P, P, P]
        L.moe_fc2_forward_fp8.argtypes = [CP, RP, P, P, P, P, P, P]
        L.moe_ffn_forward_fp8.argtypes = [CP, RP, P, P, P, P, P, P, P, P, P, P, P, P]
        L.moe_quantize_mx_fp8.argtypes = [P, I64, P, I32, P, P, P]
        L.moe_quantize_mx_fp8_weights.argtypes = [P, I64, I32, P, P, P]
        L.moe_fc1_forward_mx.argtypes = [CP, RP, P, P, P, P, P, P]
        L.moe_fc2_forward_mx.argtypes = [CP, RP, P, P, P, P, P, P]
        L.moe_ffn_forward_mx.argtypes = [CP, RP, P, P, P, P, P, P, P, P, P, P, P, P]
        for name in ("moe_route_align", "moe_fc1_forward", "moe_fc2_forward", "moe_ffn_forward",
                     "moe_combine", "moe_pack_w13", "moe_pack_w2", "moe_ffn_forward_train",
                     "moe_ffn_backward", "moe_router_backward", "moe_quantize_rows_fp8",
                     "moe_fc1_forward_fp8", "moe_fc2_forward_fp8", "moe_ffn_forward_fp8",
                     "moe_quantize_mx_fp8", "moe_quantize_mx_fp8_weights", "moe_fc1_forward_mx",
                     "moe_fc2_forward_mx", "moe_ffn_forward_mx"):
            getattr(L, name).restype = I32
        L.moe_status_string.argtypes = [I32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_launch_count.argtypes = []
        L.moe_launch_count.restype = ctypes.c_uint64
        L.moe_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        L.moe_device_error.restype = I32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoEError(fn, status)


def _q(fn: str, cfg: Config) -> int:
    v = getattr(lib(), fn)(ctypes.byref(cfg))
    if v < 0:
        raise MoEError(fn, int(v))
    return int(v)


def capacity(cfg: Config) -> int:
    return _q("moe_capacity", cfg)


def max_slots(cfg: Config) -> int:
    return _q("moe_max_slots", cfg)


def max_blocks(cfg: Config) -> int:
    return _q("moe_max_blocks", cfg)


def route_workspace_bytes(cfg: Config) -> int:
    return _q("moe_route_workspace_bytes", cfg)


def backward_workspace_bytes(cfg: Config) -> int:
    return _q("moe_backward_workspace_bytes", cfg)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def alloc_routes(cfg: Config, device) -> Routes:
    import torch
    N, K, E = max(cfg.n_tokens, 1), cfg.top_k, cfg.n_experts  # >= 1 row: non-null pointers
    S, B = max_slots(cfg), max_blocks(cfg)
    i32 = dict(dtype=torch.int32, device=device)
    return Routes(
        topk_ids=torch.empty((N, K), **i32), topk_p=torch.empty((N, K), dtype=torch.float32, device=device),
        keep=torch.empty((N, K), dtype=torch.uint8, device=device),
        expert_counts=torch.empty(E, **i32), kept_counts=torch.empty(E, **i32),
        sorted_slot_ids=torch.empty(max(S, 1), **i32), expert_ids=torch.empty(max(B, 1), **i32),
        block_start=torch.empty(E, **i32), num_tokens_post_padded=torch.empty(1, **i32),
        token_routes=torch.empty((N, K), **i32), gemm_sched=torch.zeros(4, **i32),
        slot_prob=torch.empty(max(S, 1), dtype=torch.float32, device=device))


def alloc_workspace(cfg: Config, device):
    import torch
    return torch.empty(max(route_workspace_bytes(cfg), 256), dtype=torch.uint8, device=device)


def alloc_buffers(cfg: Config, device):
    """h [S,I], o [S,H] and y [N,H] bf16 buffers for one forward."""
    import torch
    S = max(max_slots(cfg), 1)
    bf = dict(dtype=torch.bfloat16, device=device)
    return (torch.empty((S, cfg.inter), **bf), torch.empty((S, cfg.hidden), **bf),
            torch.empty((max(cfg.n_tokens, 1), cfg.hidden), **bf))


def route_align(cfg: Config, x, w_router, bias, routes: Routes, workspace, stream=None) -> None:
    rc = lib().moe_route_align(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias),
                               ctypes.byref(routes.c()), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check("moe_route_align", rc)


def fc1_forward(cfg: Config, routes: Routes, x, w13, h, stream=None) -> None:
    _check("moe_fc1_forward", lib().moe_fc1_forward(ctypes.byref(cfg), ctypes.byref(routes.c()),
                                                    _ptr(x), _ptr(w13), _ptr(h), _stream(stream)))


def fc2_forward(cfg: Config, routes: Routes, h, w2, o, stream=None) -> None:
    _check("moe_fc2_forward", lib().moe_fc2_forward(ctypes.byref(cfg), ctypes.byref(routes.c()),
                                                    _ptr(h), _ptr(w2), _ptr(o), _stream(stream)))


def ffn_forward(cfg: Config, routes: Routes, x, w13, w2, h, o, stream=None) -> None:
    _check("moe_ffn_forward", lib().moe_ffn_forward(ctypes.byref(cfg), ctypes.byref(routes.c()),
                                                    _ptr(x), _ptr(w13), _ptr(w2), _ptr(h), _ptr(o),
                                                    _stream(stream)))


def ffn_forward_train(cfg: Config, routes: Routes, x, w13, w2, h, o, preact, stream=None) -> None:
    """ffn_forward that also writes FC1's pre-activations preact [S,2I] (g | u)."""
    _check("moe_ffn_forward_train",
           lib().moe_ffn_forward_train(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(x),
                                       _ptr(w13), _ptr(w2), _ptr(h), _ptr(o), _ptr(preact),
                                       _stream(stream)))


def alloc_backward_workspace(cfg: Config, device):
    import torch
    return torch.empty(max(backward_workspace_bytes(cfg), 256), dtype=torch.uint8, device=device)


def ffn_backward(cfg: Config, routes: Routes, x, w13, w2, preact, dy, dx, dw13, dw2, dprob,
                 workspace, stream=None) -> None:
    """Expert-path backward: dx [N,H] bf16, dw13 [E,2I,H] f32, dw2 [E,H,I] f32,
    dprob [N,K] f32 (outputs overwritten)."""
    _check("moe_ffn_backward",
           lib().moe_ffn_backward(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(x), _ptr(w13),
                                  _ptr(w2), _ptr(preact), _ptr(dy), _ptr(dx), _ptr(dw13),
                                  _ptr(dw2), _ptr(dprob), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def router_backward_workspace_bytes(cfg: Config) -> int:
    return _q("moe_router_backward_workspace_bytes", cfg)


def alloc_router_backward_workspace(cfg: Config, device):
    import torch
    return torch.empty(max(router_backward_workspace_bytes(cfg), 256), dtype=torch.uint8, device=device)


def router_backward(cfg: Config, routes: Routes, x, w_router, bias, dprob, dx, dw_router, dbias,
                    workspace, stream=None, logits=None) -> None:
    """Router backward: dx += dl . W_r^T (bf16, in place), dw_router [H,E] f32 and
    dbias [E] f32 (or None) overwritten. logits: the forward's [N,E] logits
    (route_workspace_logits), or None to recompute them."""
    _check("moe_router_backward",
           lib().moe_router_backward(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(x),
                                     _ptr(w_router), _ptr(bias), _ptr(logits), _ptr(dprob),
                                     _ptr(dx), _ptr(dw_router), _ptr(dbias), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def route_workspace_logits(cfg: Config, workspace):
    """The [N,E] fp32 router logits moe_route_align left in its workspace, as a
    view of that workspace tensor."""
    import torch
    p = lib().moe_route_workspace_logits(ctypes.byref(cfg), _ptr(workspace))
    if not p:
        raise MoEError("moe_route_workspace_logits", MOE_ERR_INVALID_ARG)
    off = p - workspace.data_ptr()
    n = cfg.n_tokens * cfg.n_experts
    return workspace.view(-1)[off:off + 4 * n].view(torch.float32).view(cfg.n_tokens, cfg.n_experts)


def combine(cfg: Config, routes: Routes, o, y, stream=None) -> None:
    _check("moe_combine", lib().moe_combine(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(o),
                                            _ptr(y), _stream(stream)))


def pack_w13(cfg: Config, w_gate, w_up, w13, stream=None) -> None:
    _check("moe_pack_w13", lib().moe_pack_w13(ctypes.byref(cfg), _ptr(w_gate), _ptr(w_up),
                                              _ptr(w13), _stream(stream)))


def pack_w2(cfg: Config, w_down, w2, stream=None) -> None:
    _check("moe_pack_w2", lib().moe_pack_w2(ctypes.byref(cfg), _ptr(w_down), _ptr(w2),
                                            _stream(stream)))


def quantize_rows_fp8(m, q, scale, stream=None, rows_dev=None) -> None:
    """Row-wise E4M3 codes q [rows, cols] u8 and scales [rows] f32 of a bf16
    matrix m; rows_dev (a device int32 tensor) bounds the rows quantised."""
    rows, cols = m.shape
    _check("moe_quantize_rows_fp8",
           lib().moe_quantize_rows_fp8(_ptr(m), int(rows), _ptr(rows_dev), int(cols), _ptr(q),
                                       _ptr(scale), _stream(stream)))


def fc1_forward_fp8(cfg: Config, routes: Routes, xq, x_scale, w13q, w13_scale, h,
                    stream=None) -> None:
    _check("moe_fc1_forward_fp8",
           lib().moe_fc1_forward_fp8(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(xq),
                                     _ptr(x_scale), _ptr(w13q), _ptr(w13_scale), _ptr(h),
                                     _stream(stream)))


def fc2_forward_fp8(cfg: Config, routes: Routes, hq, h_scale, w2q, w2_scale, o,
                    stream=None) -> None:
    _check("moe_fc2_forward_fp8",
           lib().moe_fc2_forward_fp8(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(hq),
                                     _ptr(h_scale), _ptr(w2q), _ptr(w2_scale), _ptr(o),
                                     _stream(stream)))


class Fp8Weights:
    """w13 and w2 quantised row-wise once: codes (u8) and fp32 row scales."""

    def __init__(self, cfg: Config, w13, w2, stream=None):
        import torch
        E, H, I = cfg.n_experts, cfg.hidden, cfg.inter
        dev = w13.device
        self.w13q = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=dev)
        self.w13_scale = torch.empty(E * 2 * I, dtype=torch.float32, device=dev)
        self.w2q = torch.empty((E, H, I), dtype=torch.uint8, device=dev)
        self.w2_scale = torch.empty(E * H, dtype=torch.float32, device=dev)
        quantize_rows_fp8(w13.view(E * 2 * I, H), self.w13q, self.w13_scale, stream)
        quantize_rows_fp8(w2.view(E * H, I), self.w2q, self.w2_scale, stream)


def alloc_fp8_buffers(cfg: Config, device):
    """xq [N,H] u8, x_scale [N] f32, hq [S,I] u8 and h_scale [S] f32 for ffn_forward_fp8."""
    import torch
    N, S = max(cfg.n_tokens, 1), max(max_slots(cfg), 1)
    return (torch.empty((N, cfg.hidden), dtype=torch.uint8, device=device),
            torch.empty(N, dtype=torch.float32, device=device),
            torch.empty((S, cfg.inter), dtype=torch.uint8, device=device),
            torch.empty(S, dtype=torch.float32, device=device))


def ffn_forward_fp8(cfg: Config, routes: Routes, x, wq: Fp8Weights, xq, x_scale, h, hq, h_scale, o,
                    stream=None) -> None:
    """Quantise x, FC1 on FP8, quantise h, FC2 on FP8 (one C call, four launches)."""
    _check("moe_ffn_forward_fp8",
           lib().moe_ffn_forward_fp8(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(x),
                                     _ptr(wq.w13q), _ptr(wq.w13_scale), _ptr(wq.w2q),
                                     _ptr(wq.w2_scale), _ptr(xq), _ptr(x_scale), _ptr(h), _ptr(hq),
                                     _ptr(h_scale), _ptr(o), _stream(stream)))


def quantize_mx_fp8(m, q, scale, stream=None, rows_dev=None) -> None:
    """MX (block-scaled) E4M3 codes q [rows, cols] u8 and E8M0 scale codes
    [rows, cols/32] u8 of a bf16 matrix m; rows_dev bounds the rows quantised."""
    rows, cols = m.shape
    _check("moe_quantize_mx_fp8",
           lib().moe_quantize_mx_fp8(_ptr(m), int(rows), _ptr(rows_dev), int(cols), _ptr(q),
                                     _ptr(scale), _stream(stream)))


def quantize_mx_fp8_weights(m, q, scale_atoms, stream=None) -> None:
    """MX codes of packed weight rows m [rows, cols] (multiples of 128) with
    the scale bytes in the GEMMs' 512-byte atom layout."""
    rows, cols = m.shape
    _check("moe_quantize_mx_fp8_weights",
           lib().moe_quantize_mx_fp8_weights(_ptr(m), int(rows), int(cols), _ptr(q),
                                             _ptr(scale_atoms), _stream(stream)))


def fc1_forward_mx(cfg: Config, routes: Routes, xq, x_sf, w13q, w13_sf, h, stream=None) -> None:
    _check("moe_fc1_forward_mx",
           lib().moe_fc1_forward_mx(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(xq),
                                    _ptr(x_sf), _ptr(w13q), _ptr(w13_sf), _ptr(h),
                                    _stream(stream)))


def fc2_forward_mx(cfg: Config, routes: Routes, hq, h_sf, w2q, w2_sf, o, stream=None) -> None:
    _check("moe_fc2_forward_mx",
           lib().moe_fc2_forward_mx(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(hq),
                                    _ptr(h_sf), _ptr(w2q), _ptr(w2_sf), _ptr(o), _stream(stream)))


class MxWeights:
    """w13 and w2 MX-quantised once: E4M3 codes and E8M0 block scales in the
    GEMMs' atom layout."""

    def __init__(self, cfg: Config, w13, w2, stream=None):
        import torch
        E, H, I = cfg.n_experts, cfg.hidden, cfg.inter
        dev = w13.device
        self.w13q = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=dev)
        self.w13_sf = torch.empty(E * 2 * I * H // 32, dtype=torch.uint8, device=dev)
        self.w2q = torch.empty((E, H, I), dtype=torch.uint8, device=dev)
        self.w2_sf = torch.empty(E * H * I // 32, dtype=torch.uint8, device=dev)
        quantize_mx_fp8_weights(w13.view(E * 2 * I, H), self.w13q, self.w13_sf, stream)
        quantize_mx_fp8_weights(w2.view(E * H, I), self.w2q, self.w2_sf, stream)


def alloc_mx_buffers(cfg: Config, device):
    """xq [N,H] u8, x_sf [N,H/32] u8, hq [S,I] u8 and h_sf [S,I/32] u8 for ffn_forward_mx."""
    import torch
    N, S = max(cfg.n_tokens, 1), max(max_slots(cfg), 1)
    u8 = dict(dtype=torch.uint8, device=device)
    return (torch.empty((N, cfg.hidden), **u8), torch.empty((N, cfg.hidden // 32), **u8),
            torch.empty((S, cfg.inter), **u8), torch.empty((S, cfg.inter // 32), **u8))


def ffn_forward_mx(cfg: Config, routes: Routes, x, wq: MxWeights, xq, x_sf, h, hq, h_sf, o,
                   stream=None) -> None:
    """Quantise x, FC1 on MX operands, quantise h, FC2 on MX (one C call, four launches)."""
    _check("moe_ffn_forward_mx",
           lib().moe_ffn_forward_mx(ctypes.byref(cfg), ctypes.byref(routes.c()), _ptr(x),
                                    _ptr(wq.w13q), _ptr(wq.w13_sf), _ptr(wq.w2q), _ptr(wq.w2_sf),
                                    _ptr(xq), _ptr(x_sf), _ptr(h), _ptr(hq), _ptr(h_sf), _ptr(o),
                                    _stream(stream)))


def forward(cfg: Config, x, w_router, bias, w13, w2, routes: Routes, workspace, h, o, y,
            stream=None) -> None:
    """The whole layer: route_align, ffn_forward, combine (three C calls)."""
    route_align(cfg, x, w_router, bias, routes, workspace, stream)
    ffn_forward(cfg, routes, x, w13, w2, h, o, stream)
    combine(cfg, routes, o, y, stream)


def launch_count() -> int:
    return int(lib().moe_launch_count())


def device_error() -> int:
    v = ctypes.c_uint32(0)
    _check("moe_device_error", lib().moe_device_error(ctypes.byref(v)))
    return int(v.value)


def ladder_pick(buckets, n: int, max_pad_ratio: float = 0.0) -> int:
    """Index of the bucket a batch of n tokens replays, or -1 for eager."""
    arr = (ctypes.c_int32 * len(buckets))(*buckets)
    return int(lib().moe_ladder_pick(ctypes.cast(arr, ctypes.c_void_p), len(buckets), int(n),
                                     float(max_pad_ratio)))


class Ladder:
    """Captured forward graphs at a ladder of token-count buckets (moe_ladder_*).
    Allocates the layer's buffers for the top bucket (cfg.n_tokens must equal
    the last bucket); x, y, routes, h, o are torch tensors sized for it. A
    forward of n tokens reads x[:n] and writes y[:n]."""

    def __init__(self, cfg: Config, buckets, max_pad_ratio, w_router, bias, w13, w2, device):
        import torch
        self.cfg, self.buckets = cfg, list(buckets)
        dev = torch.device(device)
        N, H = cfg.n_tokens, cfg.hidden
        self.x = torch.zeros((max(N, 1), H), dtype=torch.bfloat16, device=dev)
        self.routes = alloc_routes(cfg, dev)
        self.ws = alloc_workspace(cfg, dev)
        self.h, self.o, self.y = alloc_buffers(cfg, dev)
        self.n_valid = torch.zeros(1, dtype=torch.int32, device=dev)
        self._keep = (w_router, bias, w13, w2)  # the graphs hold their addresses
        self._bufs = _LayerBufsC(self.x.data_ptr(), w_router.data_ptr(), _ptr(bias), w13.data_ptr(),
                                 w2.data_ptr(), self.routes.c(), self.ws.data_ptr(),
                                 self.ws.numel(), self.h.data_ptr(), self.o.data_ptr(),
                                 self.y.data_ptr(), self.n_valid.data_ptr())
        arr = (ctypes.c_int32 * len(self.buckets))(*self.buckets)
        handle = ctypes.c_void_p()
        _check("moe_ladder_create",
               lib().moe_ladder_create(ctypes.byref(cfg), ctypes.cast(arr, ctypes.c_void_p),
                                       len(self.buckets), float(max_pad_ratio),
                                       ctypes.byref(self._bufs), ctypes.byref(handle)))
        self._h = handle

    def forward(self, n: int, stream=None) -> int:
        """One forward of x[:n]; returns the bucket index replayed, -1 for eager."""
        b = ctypes.c_int(0)
        _check("moe_ladder_forward", lib().moe_ladder_forward(self._h, int(n), _stream(stream),
                                                              ctypes.byref(b)))
        return b.value

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().moe_ladder_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
