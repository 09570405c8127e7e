"""Host logic of bench.py without a GPU: max-over-ranks timing with two gloo
ranks, the algorithmic work model, and the roofline arithmetic."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, l = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, dist)
    q.put((r, slowest))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_single_process_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_work_model_counts():
    w = synth.WORKLOADS["dsv3"]
    kc = np.full(256, 130)
    kc[:6] = 0
    m = bench.work_model(w, kc)
    assert m["_active"] == 250 and m["_kept"] == 250 * 130
    rows = 250 * 144
    assert m["fc1"]["bytes"] == 250 * 2 * 2048 * 7168 * 2 + 4096 * 7168 * 2 + rows * 2048 * 2
    assert m["fc2"]["flops"] == 2.0 * 250 * 130 * 2048 * 7168


def test_roofline_picks_the_binding_resource():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 1000.0, "sm_max_mhz": 2000.0, "_source": "test"}
    model = {"fc1": {"bytes": 1e9, "flops": 1e12, "units": 1}}  # 1 ms of HBM, 1 ms of tensor
    model["fc1"]["flops"] = 0.5e12                               # now HBM binds
    r = bench.roofline_for("fc1", model, 2.0, peaks, "x")
    assert r["bound"] == "hbm" and abs(r["achieved"] - 500.0) < 1e-9 and abs(r["frac"] - 0.5) < 1e-12
    model["fc1"]["flops"] = 4e12                                 # tensor binds
    r = bench.roofline_for("fc1", model, 8.0, peaks, "x")
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-12


def test_activation_variant_options():
    """--activation / --prob-in-act reach the layer config and the JSON config
    keys; the FP8 line keeps the default layer, so combining them is refused."""
    a = bench.parse_args([])
    assert bench.act_code(a) == 0 and bench.variant_config(a) == {}
    a = bench.parse_args(["--activation", "geglu", "--prob-in-act"])
    assert bench.act_code(a) == 1
    assert bench.variant_config(a) == {"activation": "geglu", "prob_in_act": True}
    with pytest.raises(SystemExit):
        bench.parse_args(["--fp8", "--activation", "geglu"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--fp8", "--prob-in-act"])
