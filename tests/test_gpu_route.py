"""Routing on the GPU against the oracle, bit for bit: top-K ids, renormalised
probabilities, per-expert counts, drop set and the whole route-list layout."""
import numpy as np
import pytest

import synth
from gpu_util import Problem, assert_routing_equal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "qwen3_small", "qwen3_30b", "dsv3"])
@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_route_align_bit_exact_full_size(name, bm):
    w = synth.WORKLOADS[name]
    P = Problem(w, bm=bm, host_weights=False, with_ffn=False)
    P.run()
    assert_routing_equal(P, P.oracle_routing())


def _w(N, H, E, K, I=128, cn=1, cd=1, **kw):
    return synth.Workload("case", N, H, E, K, I, cn, cd, **kw)


@pytest.mark.parametrize("w,bm", [
    (_w(1, 128, 8, 2), 16),            # one token
    (_w(31, 128, 8, 2), 16),           # one ragged 32-token chunk
    (_w(33, 128, 8, 2), 32),           # the second chunk holds one token
    (_w(63, 128, 8, 2), 16),           # ragged second chunk
    (_w(65, 256, 16, 4, cn=1, cd=2), 32),  # three chunks, the last holds one token; heavy drops
    (_w(130, 128, 1, 1), 16),          # one expert
    (_w(97, 128, 5, 5), 64),           # K = E: every expert picked
    (_w(200, 128, 256, 16), 16),       # widest supported router
    (_w(300, 384, 12, 3, cn=7, cd=1), 128),  # capacity above N: nothing dropped
    (_w(0, 128, 8, 2), 16),            # empty batch
    (_w(24576, 128, 8, 2), 32),        # the largest supported token count
    (_w(24576, 128, 64, 6, cn=0, cd=1, zipf_s=0.8, ladder=(2, 4), ladder_den=2), 32),  # dropless
    # each form of the logits kernel at a size past the few-chains bound:
    (_w(4096, 1024, 16, 4, cn=5, cd=4), 32),   # E < 32: one thread per token and expert pair
    (_w(2048, 256, 31, 3), 16),                # odd E: the same, scalar W_r loads
    (_w(4096, 2048, 32, 4), 32),               # 32-expert tiles, TMA stages of 32
    (_w(3000, 4096, 64, 6, cn=5, cd=4), 64),   # 64-expert tiles, TMA stages of 64
    (_w(3000, 512, 48, 4), 32),                # E below the 64-wide tile: cp.async form
    (_w(2500, 256, 130, 6), 32),               # E not a multiple of 4: cp.async form, 4-byte W_r loads
])
def test_route_align_edge_shapes(w, bm):
    P = Problem(w, bm=bm, host_weights=False, with_ffn=False)
    P.run()
    assert_routing_equal(P, P.oracle_routing())


def test_identical_tokens_ties_go_to_lower_token():
    """Every token the same: equal probabilities across tokens, so each
    expert keeps its lowest token indices."""
    w = _w(256, 128, 8, 2, cn=1, cd=2)
    row = synth.normal_bf16_bits(0, 0, 0, 128)
    P = Problem(w, bm=16, host_weights=False, x_bits=np.tile(row, (256, 1)), with_ffn=False)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    e0 = R.topk_ids[0, 0]
    assert list(R.layout.sorted_slot_ids[e0 * R.layout.cpad:e0 * R.layout.cpad + 4]) == [0, 1, 2, 3]


def test_bias_and_no_renorm():
    w = _w(500, 256, 32, 4, cn=3, cd=4)
    bias = (np.random.default_rng(0).standard_normal(32) * 2).astype(np.float32)
    P = Problem(w, bm=32, host_weights=False, bias=bias, renorm=0, with_ffn=False)
    P.run()
    assert_routing_equal(P, P.oracle_routing())


def test_zero_logits_all_ties():
    """Zero router weight: every probability equal, every tie rule exercised."""
    w = _w(130, 128, 8, 3, cn=1, cd=2, wr_std=0.0)
    P = Problem(w, bm=16, host_weights=False, with_ffn=False)
    P.run()
    R = P.oracle_routing()
    assert_routing_equal(P, R)
    assert np.all(R.topk_ids == np.array([0, 1, 2]))
