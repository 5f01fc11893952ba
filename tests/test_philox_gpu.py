"""GPU noise generator (drs_philox_gumbel) against the oracle: the words bit
for bit, the Gumbel values within GUMBEL_ABS."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import drs
from parity import GUMBEL_ABS

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,row0,rows,vocab", [
    (0, 0, 64, 1000),
    (0x123456789ABCDEF0, 5, 33, 4099),
    (2**64 - 1, 2**32 - 3, 7, 257),     # rows crossing the 32-bit boundary
    (7, 123456789012, 3, 5),
])
def test_noise_matches_oracle(seed, row0, rows, vocab):
    lib = drs()
    bits, g = lib.philox_gumbel(seed, row0, rows, vocab)
    torch.cuda.synchronize()
    rb, rg = oracle.philox_gumbel(seed, row0, rows, vocab)
    assert np.array_equal(bits.cpu().numpy().view(np.uint32), rb)
    assert np.max(np.abs(g.cpu().numpy().astype(np.float64) - rg)) <= GUMBEL_ABS


def test_noise_extremes():
    """The fp32 Gumbel of the extreme words: u = 1e-20 and u = 1 - 2^-24."""
    lib = drs()
    bits, g = lib.philox_gumbel(3, 0, 512, 4096)
    b = bits.cpu().numpy().view(np.uint32).ravel()
    gv = g.cpu().numpy().ravel()
    ref = np.array([oracle.gumbel_of_bits(int(x)) for x in b[:20000]])
    assert np.max(np.abs(gv[:20000] - ref)) <= GUMBEL_ABS
    assert gv.max() <= 16.64 and gv.min() >= -3.84
