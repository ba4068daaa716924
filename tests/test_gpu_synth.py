"""The seeded input generator: its CUDA implementation gives the numpy implementation's bits.

Every large parity input (the B=8 T=2048 workloads, the 36 GB decode pool) is generated on the
device, and the oracle's copy of any sampled slice is regenerated on the host; both sides must
therefore agree exactly, element for element, in fp32 and in bf16, at any offset into a stream."""
import numpy as np
import pytest
import torch

import glasynth as gs
from glasynth import device as gdev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sigma", [1.0, float(1 / np.sqrt(96.0)), 0.1, 0.01])
@pytest.mark.parametrize("start", [0, 12345, (1 << 33) + 7])
def test_device_generator_matches_host_bitwise(sigma, start):
    n = 1 << 20
    host = gs.normal(9, 5, (n,), sigma, start=start)
    dev32 = gdev.normal((n,), 9, 5, sigma, torch.float32, "cuda", start=start).cpu().numpy()
    assert np.array_equal(dev32.view(np.uint32), host.view(np.uint32))
    dev16 = gdev.normal((n,), 9, 5, sigma, torch.bfloat16, "cuda", start=start)
    assert np.array_equal(dev16.view(torch.int16).cpu().numpy().astype(np.uint16), gs.bf16_bits(host))


def test_device_generator_rows_match_host_rows():
    """normal_rows regenerates sampled rows of a device-generated tensor (the decode pool's way)."""
    t = gdev.normal((64, 16, 96), 2, 7, 0.1, torch.float32, "cuda").cpu().numpy()
    rows = gs.normal_rows(2, 7, (96,), [0, 5 * 16 + 3, 63 * 16 + 15], 0.1)
    assert np.array_equal(rows[0], t[0, 0]) and np.array_equal(rows[1], t[5, 3])
    assert np.array_equal(rows[2], t[63, 15])
