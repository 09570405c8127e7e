"""Host side of the seeded input generator (no MoE arithmetic here)."""
import numpy as np
import pytest
from scipy import stats

import synth


def test_counter_based_slices_agree():
    full = synth.normal_f32(0, 2, 0, 5000, 0.02)
    part = synth.normal_f32(0, 2, 1234, 777, 0.02)
    assert np.array_equal(full[1234:1234 + 777], part)
    assert not np.array_equal(synth.normal_f32(0, 3, 0, 100), synth.normal_f32(0, 2, 0, 100))
    assert not np.array_equal(synth.normal_f32(1, 2, 0, 100), synth.normal_f32(0, 2, 0, 100))


@pytest.mark.parametrize("seed,stream,start,count,std", [
    (0, 0, 0, 200_000, 1.0), (0, 2, 123_456_789, 50_000, 0.02), (3, 4, 10 ** 11, 50_000, 0.006)])
def test_c_twin_matches_numpy_definition(seed, stream, start, count, std):
    ref = synth.normal_f32_numpy(seed, stream, start, count, std)
    assert np.array_equal(synth.normal_f32(seed, stream, start, count, std).view(np.uint32),
                          ref.view(np.uint32))
    assert np.array_equal(synth.normal_bf16_bits(seed, stream, start, count, std),
                          synth.f32_to_bf16_bits(ref))


def test_normal_statistics():
    v = synth.normal_f32(0, 0, 0, 400000).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    assert stats.kstest(v, "norm").pvalue > 1e-3
    assert abs(stats.kurtosis(v)) < 0.05


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.00390625, 1.005859375, 1.0078125, -2.5, 3.0e-3], np.float32)
    # 1+2^-8 is halfway between 1 and 1+2^-7: ties to even (1.0);
    # 1+1.5*2^-8 is above halfway: rounds up to 1+2^-7
    b = synth.f32_to_bf16_bits(f)
    back = synth.bf16_bits_to_f32(b)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0078125 and back[3] == 1.0078125
    assert back[4] == -2.5
    assert abs(back[5] - 3.0e-3) <= 2 ** -8 * 3.0e-3  # half an ulp: 2^-8 relative


def test_zipf_bias_is_minus_s_log_rank():
    b = synth.zipf_bias(0, 128, 1.0)
    ranks = np.rint(np.exp(-b.astype(np.float64))).astype(int)
    assert sorted(ranks.tolist()) == list(range(1, 129))
    assert b.max() == 0.0
    b8 = synth.zipf_bias(0, 128, 0.8)
    assert np.allclose(b8, 0.8 * b, rtol=1e-6)
