"""The Zipf-skewed workloads' router bias (input recipe, CPU).

The Qwen3-30B-A3B-shaped layer asks for a router bias "drawn so expert
popularity follows Zipf(s=1.0)", the dropless layer for "skewed Zipf(s=0.8)
routing". The stored biases (synth/data, written by
oracle/calibrate_router_bias.py from a calibration batch of its own stream)
must give, on the batches the tests and the benchmark use, route shares that
follow the capped Zipf target up to the binomial spread of one batch.
"""
import numpy as np
import pytest

import oracle
import synth


def test_target_shares_closed_form():
    # Zipf(1) over 128 experts with top-8: the head share 1/H_128 = 0.184 is
    # above 1/8, so rank 1 is capped at 1/8 and the other ranks share 7/8 in
    # proportion to 1/r
    t = synth.zipf_target_shares(128, 8, 1.0)
    assert abs(t.sum() - 1.0) < 1e-12
    assert t[0] == pytest.approx(1 / 8, rel=1e-12)
    h2 = sum(1.0 / r for r in range(2, 129))
    for r in (2, 3, 10, 64, 128):
        assert t[r - 1] == pytest.approx((7 / 8) * (1.0 / r) / h2, rel=1e-12)
    # Zipf(0.8) over 64 experts with top-6: the head share 1/sum r^-0.8 is
    # below 1/6, so nothing is capped
    t8 = synth.zipf_target_shares(64, 6, 0.8)
    z = np.arange(1, 65, dtype=np.float64) ** -0.8
    assert np.allclose(t8, z / z.sum(), rtol=1e-12, atol=0)
    assert t8[0] < 1 / 6
    # a cap that binds twice: Zipf(2) over 16 experts with top-4
    t2 = synth.zipf_target_shares(16, 4, 2.0)
    assert abs(t2.sum() - 1.0) < 1e-12 and t2.max() <= 0.25 * (1 + 1e-12)
    unc = t2 < 0.25 * (1 - 1e-12)
    r = np.arange(1, 17)[unc]
    assert np.allclose(t2[unc] * r ** 2, (t2[unc] * r ** 2)[0], rtol=1e-12)


@pytest.mark.parametrize("name", ["qwen3_30b", "dropless", "dropless_e16"])
def test_stored_bias_loads(name):
    w = synth.WORKLOADS[name]
    b = synth.router_bias(w)
    assert b.dtype == np.float32 and b.shape == (w.n_experts,) and np.isfinite(b).all()
    ranks = synth.zipf_ranks(w.seed, w.n_experts)
    assert b[np.argmin(ranks)] == 0.0
    # more popular ranks carry a larger bias, with a few local exceptions
    # where an expert's router column already favours it
    rho = np.corrcoef(np.argsort(np.argsort(b)), -ranks)[0, 1]
    assert rho > 0.9


@pytest.mark.parametrize("name,n", [("qwen3_30b", 8192), ("dropless", 16384), ("dropless", 4096)])
def test_route_shares_follow_zipf(name, n):
    w = synth.WORKLOADS[name].with_tokens(n)
    E, K, H = w.n_experts, w.top_k, w.hidden
    inp = synth.make_host_inputs(w, experts=[])
    ids, _, _, _ = oracle.router(inp["x"], inp["wr"], inp["bias"], K)
    share = np.bincount(ids.ravel(), minlength=E) / ids.size
    ranks = synth.zipf_ranks(w.seed, E)
    target = synth.zipf_target_shares(E, K, w.zipf_s)[ranks - 1]
    # binomial spread of one batch: expert e is picked by each of the n
    # tokens independently with probability q = K * target
    q = np.minimum(K * target, 1.0)
    sigma = np.sqrt(n * q * (1 - q)) / (n * K)
    capped = q >= 1.0
    assert (share[capped] >= 0.99 * target[capped]).all()
    z = np.abs(share - target)[~capped] / sigma[~capped]
    assert z.max() < 4.0, z.max()
    if n >= 8192:
        by_rank = np.empty(E)
        by_rank[ranks - 1] = np.abs(share / target - 1.0)
        assert (by_rank[:64] <= 0.10).sum() >= 58
