"""The device twin of the input generator gives the host generator's bits."""
import numpy as np
import pytest
import torch

import synth
import synth.gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("stream,std,index0", [(0, 1.0, 0), (2, 0.02, 0), (4, 0.006, 10 ** 10)])
def test_gpu_generator_matches_host_bits(stream, std, index0):
    n = 300_000
    host = synth.normal_f32(0, stream, index0, n, std)
    t32 = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.gpu.fill(t32, 0, stream, std, index0=index0)
    assert np.array_equal(t32.cpu().numpy().view(np.uint32), host.view(np.uint32))
    tb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    synth.gpu.fill(tb, 0, stream, std, index0=index0)
    assert np.array_equal(tb.cpu().view(torch.int16).numpy().view(np.uint16),
                          synth.f32_to_bf16_bits(host))


def test_gpu_generator_permuted_layout():
    """dims/strides fill: a transposed view takes the logical indices."""
    R, C = 96, 160
    host = synth.normal_f32(0, 3, 0, R * C).reshape(R, C)
    t = torch.empty((C, R), dtype=torch.float32, device="cuda")
    synth.gpu.fill(t, 0, 3, 1.0, dims=(1, C, R), strides=(0, 1, C))
    assert np.array_equal(t.cpu().numpy(), host.T)
