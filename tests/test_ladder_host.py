"""Bucket choice of the graph ladder (host logic, no GPU): the first bucket at
or above the batch size, eager above the top bucket or past the padding ratio
("[4/5] feat: capture the FFN experts at bucketed padded shapes", What this
adds)."""
import pytest

import mixture_experts_routing_gb300 as moe


@pytest.mark.parametrize("n,ratio,want", [
    (0, 0.0, 0), (1, 0.0, 0), (256, 0.0, 0), (257, 0.0, 1), (2048, 0.0, 3), (2049, 0.0, -1),
    (1, 2.0, -1), (200, 2.0, 0), (127, 2.0, -1), (300, 1.5, -1), (400, 1.5, 1), (1500, 1.5, 3),
    (1024, 1.0, 2), (1025, 1.0, -1),
])
def test_ladder_pick(n, ratio, want):
    assert moe.ladder_pick([256, 512, 1024, 2048], n, ratio) == want


def test_ladder_pick_rejects_bad_input():
    assert moe.ladder_pick([256], -1) == -1
    assert moe.ladder_pick([], 5) == -1
