"""The device filler of the seeded inputs writes the same bits as the host filler."""
import numpy as np
import pytest

import synth
from _util import host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,tid,offset,sigma", [(1 << 20, 5, 0, 0.02), (100003, 77, 123456789, 1.0),
                                                (4096, synth.W_G, 383 * 2048 * 7168, 0.02)])
def test_device_filler_matches_host(n, tid, offset, sigma):
    import torch
    t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    synth.fill_bf16_dev(t.data_ptr(), n, 0, tid, offset, sigma)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(t), synth.bf16(n, 0, tid, offset, sigma))
    f = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.fill_f32_dev(f.data_ptr(), n, 0, tid, offset, sigma)
    torch.cuda.synchronize()
    assert np.array_equal(f.cpu().numpy().view(np.uint32), synth.f32(n, 0, tid, offset, sigma).view(np.uint32))
