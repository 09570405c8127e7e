"""moe_route_align_noalloc: the routing entry point for callers that cannot
allocate device memory (a plugin inside another runtime that owns every
allocation, a serving loop that bans cudaMalloc because it can synchronise
the device, a fixed up-front memory budget). It must give exactly what
moe_route_align gives with a caller-provided workspace, call after call, even
though every call reuses the same built-in scratch array. This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_routing_gb300 as moe
import synth
from gpu_util import Problem

pytestmark = pytest.mark.gpu


def _noalloc(cfg, x, wr, bias, routes):
    L = moe.lib()
    f = L.moe_route_align_noalloc
    f.argtypes = [ctypes.POINTER(moe.Config), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.POINTER(moe._RoutesC), ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(ctypes.byref(cfg), x.data_ptr(), wr.data_ptr(),
             None if bias is None else bias.data_ptr(), ctypes.byref(routes.c()),
             torch.cuda.current_stream().cuda_stream)


def _snapshot(routes):
    return {n: getattr(routes, n).clone() for n, _ in moe.Routes.FIELDS}


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # Zipf-routed workload: hot experts overflow their capacity, so the drop
    # set and the layout depend on every scratch region being right.
    P = Problem(synth.WORKLOADS["qwen3_30b"], bm=32, with_ffn=False)
    assert moe.route_workspace_bytes(P.cfg) <= 8 << 20
    x2 = torch.from_numpy(synth.normal_bf16_bits(7, 0, 0, P.w.n_tokens * P.w.hidden)
                          .reshape(P.w.n_tokens, P.w.hidden).view(np.int16)).view(torch.bfloat16).to(P.dev)
    for x in (P.x, x2):  # the second call finds the first call's data in the scratch
        moe.route_align(P.cfg, x, P.wr_d, P.bias_d, P.routes, P.ws)
        torch.cuda.synchronize()
        want = _snapshot(P.routes)
        for n, _ in moe.Routes.FIELDS:  # poison, so a field left unwritten shows up
            getattr(P.routes, n).fill_(-7 if getattr(P.routes, n).dtype != torch.uint8 else 77)
        assert _noalloc(P.cfg, x, P.wr_d, P.bias_d, P.routes) == 0
        torch.cuda.synchronize()
        for n, _ in moe.Routes.FIELDS:
            assert torch.equal(getattr(P.routes, n), want[n]), n
    assert moe.device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    cfg = moe.Config(24576, 128, 256, 8, 128, 1, 1, block_m=32)  # 24 MiB of logits alone
    assert moe.route_workspace_bytes(cfg) > 8 << 20
    P = Problem(synth.Workload("small", 64, 128, 8, 2, 128, 1, 1), bm=32, with_ffn=False)
    assert _noalloc(cfg, P.x, P.wr_d, None, P.routes) == -3  # MOE_ERR_WORKSPACE, nothing launched
