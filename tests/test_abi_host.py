"""The C ABI without a GPU: the library loads, exports every entry point that
include/moe.h declares, answers size queries, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

import mixture_experts_routing_gb300 as moe
import oracle
import synth
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\**\s+\**(moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    from mixture_experts_routing_gb300 import _build
    _build.build()
    return moe.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route_align", "moe_ffn_forward", "moe_combine", "moe_fc1_forward",
              "moe_fc2_forward", "moe_pack_w13", "moe_pack_w2", "moe_route_workspace_bytes",
              "moe_max_slots", "moe_capacity", "moe_status_string", "moe_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def _cfg(w, bm=32):
    return moe.Config(w.n_tokens, w.hidden, w.n_experts, w.top_k, w.inter, w.cap_num, w.cap_den,
                      block_m=bm)


@pytest.mark.parametrize("name", ["tiny", "qwen3_small", "qwen3_30b", "dsv3"])
@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_size_queries_match_oracle_capacity(L, name, bm):
    w = synth.WORKLOADS[name]
    cfg = _cfg(w, bm)
    cap = oracle.capacity(w.n_tokens, w.top_k, w.n_experts, w.cap_num, w.cap_den)
    assert moe.capacity(cfg) == cap
    cpad = -(-cap // bm) * bm
    assert moe.max_slots(cfg) == w.n_experts * cpad
    assert moe.max_blocks(cfg) == w.n_experts * cpad // bm
    assert moe.route_workspace_bytes(cfg) >= 4 * w.n_tokens * w.n_experts


def test_invalid_configs_fail_closed(L):
    good = dict(n_tokens=64, hidden=128, n_experts=8, top_k=2, inter=128, cap_num=1, cap_den=1,
                block_m=32)
    bad_fields = [("n_tokens", -1), ("hidden", 0), ("n_experts", 0), ("top_k", 0), ("top_k", 9),
                  ("cap_den", 0), ("block_m", 8), ("block_m", 48)]
    for k, v in bad_fields:
        c = moe.Config(**dict(good, **{k: v}))
        assert L.moe_max_slots(ctypes.byref(c)) == -1, (k, v)
    unsupported = [("hidden", 192), ("inter", 64), ("n_experts", 300), ("n_tokens", 10 ** 6)]
    for k, v in unsupported:
        c = moe.Config(**dict(good, **{k: v}, top_k=2))
        assert L.moe_max_slots(ctypes.byref(c)) == -2, (k, v)
    assert L.moe_max_slots(None) == -1
    # the token bound of the route kernels: 24576 is accepted, one more is not
    c = moe.Config(**dict(good, n_tokens=24576))
    assert L.moe_max_slots(ctypes.byref(c)) > 0
    c = moe.Config(**dict(good, n_tokens=24577))
    assert L.moe_max_slots(ctypes.byref(c)) == -2


def test_entry_points_reject_bad_arguments_before_launch(L):
    cfg = moe.Config(64, 128, 8, 2, 128, 1, 1, block_m=32)
    empty = moe._RoutesC()
    # missing routes
    assert L.moe_route_align(ctypes.byref(cfg), 16, 16, None, ctypes.byref(empty), 256, 1 << 20,
                             None) == -1
    full = moe._RoutesC(*([256] * len(moe._RoutesC._fields_)))
    # null x / router weight
    assert L.moe_route_align(ctypes.byref(cfg), None, 16, None, ctypes.byref(full), 256, 1 << 20,
                             None) == -1
    # misaligned x
    assert L.moe_route_align(ctypes.byref(cfg), 18, 16, None, ctypes.byref(full), 256, 1 << 20,
                             None) == -1
    # workspace missing / too small
    assert L.moe_route_align(ctypes.byref(cfg), 16, 16, None, ctypes.byref(full), None, 1 << 20,
                             None) == -3
    need = moe.route_workspace_bytes(cfg)
    assert L.moe_route_align(ctypes.byref(cfg), 16, 16, None, ctypes.byref(full), 256, need - 1,
                             None) == -3
    # GEMMs and combine: null / misaligned operands
    assert L.moe_fc1_forward(ctypes.byref(cfg), ctypes.byref(full), None, 256, 256, None) == -1
    assert L.moe_fc2_forward(ctypes.byref(cfg), ctypes.byref(full), 256, 264, 256, None) == -1
    assert L.moe_combine(ctypes.byref(cfg), ctypes.byref(full), 256, None, None) == -1
    assert L.moe_combine(ctypes.byref(cfg), None, 256, 256, None) == -1
    assert L.moe_pack_w13(ctypes.byref(cfg), None, 256, 256, None) == -1
    assert L.moe_pack_w2(ctypes.byref(cfg), 256, None, None) == -1
    bad = moe.Config(64, 100, 8, 2, 128, 1, 1, block_m=32)
    assert L.moe_combine(ctypes.byref(bad), ctypes.byref(full), 256, 256, None) == -2


def test_status_strings(L):
    assert moe.status_string(0) == "ok"
    assert "unsupported" in moe.status_string(-2)
    assert moe.status_string(12345) == "unknown status"


@pytest.mark.parametrize("N", [128, 1000, 16384])
def test_dropless_sizes_match_oracle_bound(L, N):
    ladder = [2, 3, 4, 5, 6, 8]  # 0.5x .. 2x of the expected rows per expert
    cfg = moe.Config(N, 4096, 64, 6, 1408, 0, 1, block_m=32, ladder=ladder, ladder_den=4)
    assert moe.capacity(cfg) == N
    want = oracle.dropless_s_max(N, 6, 64, 32, ladder, 4)
    assert moe.max_slots(cfg) == -(-want // 32) * 32
    assert moe.max_blocks(cfg) * 32 == moe.max_slots(cfg)


def test_dropless_ladder_validation(L):
    base = dict(n_tokens=64, hidden=128, n_experts=8, top_k=2, inter=128, cap_num=0, cap_den=1)
    ok = moe.Config(**base, ladder=[1, 2, 4], ladder_den=2)
    assert L.moe_max_slots(ctypes.byref(ok)) > 0
    for lad, den in (([4, 2], 2), ([0, 1], 2), ([1, 2], 0), (list(range(1, 18)), 1)):
        c = moe.Config(**base, ladder=lad, ladder_den=den)
        assert L.moe_max_slots(ctypes.byref(c)) == -1, (lad, den)
    no_ladder = moe.Config(**base)
    assert moe.max_slots(no_ladder) == 64 * 2 + 8 * 32


def test_router_backward_rejects_bad_arguments_before_launch(L):
    """Argument checks of moe_router_backward run on the host before any
    device work: routes, operands, 16-byte alignment of x and dx, workspace."""
    cfg = moe.Config(64, 128, 8, 2, 128, 1, 1, block_m=32)
    full = moe._RoutesC(*([256] * len(moe._RoutesC._fields_)))
    need = L.moe_router_backward_workspace_bytes(ctypes.byref(cfg))
    assert need > 0

    def call(routes=ctypes.byref(full), x=256, wr=256, dprob=256, dx=256, dwr=256, ws=256,
             nbytes=None):
        return L.moe_router_backward(ctypes.byref(cfg), routes, x, wr, None, None, dprob, dx, dwr,
                                     None, ws, need if nbytes is None else nbytes, None)

    assert call(routes=None) == -1
    assert call(wr=None) == -1
    assert call(dwr=None) == -1
    assert call(dprob=None) == -1
    assert call(x=264) == -1 and call(x=258) == -1   # x not 16-byte aligned
    assert call(dx=264) == -1                        # dx not 16-byte aligned
    assert call(ws=None) == -3 and call(nbytes=need - 1) == -3 and call(ws=264) == -3
