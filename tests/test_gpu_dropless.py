"""Dropless, bucketed layout on the GPU against the oracle: routing and route
list bit-exact (ladder extents, dynamic block_start, device-side padded
extent), FFN and combine within tolerance."""
import numpy as np
import pytest

import synth
from gpu_util import (Problem, assert_close, assert_routing_equal, check_combine_property,
                      check_expert_slots)
import oracle

pytestmark = pytest.mark.gpu

DL = synth.WORKLOADS["dropless"]


@pytest.mark.parametrize("N", list(DL.sweep))
def test_dropless_route_align_bit_exact_sweep(N):
    P = Problem(DL.with_tokens(N), bm=32, host_weights=False, with_ffn=False)
    P.run()
    assert_routing_equal(P, P.oracle_routing())


@pytest.mark.parametrize("bm", [16, 64, 128])
def test_dropless_route_align_block_sizes(bm):
    P = Problem(DL.with_tokens(3000), bm=bm, host_weights=False, with_ffn=False)
    P.run()
    assert_routing_equal(P, P.oracle_routing())


def test_dropless_without_ladder_pads_to_blocks():
    w = synth.Workload("noladder", 777, 128, 12, 3, 128, 0, 1, zipf_s=1.2)
    P = Problem(w, bm=32, host_weights=False, with_ffn=False)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    assert np.array_equal(np.diff(np.append(R.layout.block_start, 0))[:-1] * 32,
                          (R.layout.expert_counts[:-1] + 31) // 32 * 32)


@pytest.mark.parametrize("w,bm", [
    (synth.Workload("dl_small", 300, 256, 8, 3, 256, 0, 1, zipf_s=0.8, ladder=(2, 3, 4, 5, 6, 8),
                    ladder_den=4), 32),
    (synth.Workload("dl_hot", 640, 128, 6, 2, 384, 0, 1, zipf_s=2.0, ladder=(1, 2), ladder_den=2), 16),
])
def test_dropless_forward_small_elementwise(w, bm):
    P = Problem(w, bm=bm, host_weights=True)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    W = P.expert_weights(range(w.n_experts))
    y_ref = oracle.forward_tokens(0, w.n_tokens, P.x_bits, W, w.hidden, w.inter, R.topk_ids,
                                  R.topk_p, R.layout.keep)
    assert_close(P.y.float().cpu().numpy()[:w.n_tokens], y_ref, "y")
    check_expert_slots(P, R, range(w.n_experts))
    check_combine_property(P, R)


def test_dropless_forward_full_size_sampled():
    """N = 16384: the hottest expert holds several 256-slot tiles."""
    P = Problem(DL, bm=32, host_weights=False)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    kc = R.layout.kept_counts
    order = np.argsort(kc, kind="stable")
    experts = sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2])})
    check_expert_slots(P, R, experts)
    check_combine_property(P, R)
