"""The temperature quotient of the kernels (drs_scaled_logits) against IEEE
fp32 division, bit for bit, over every fp32 input and a set of temperatures
that includes the workloads' and reciprocal-rounding worst cases."""
import numpy as np
import pytest
import torch

from gpu_util import drs

pytestmark = pytest.mark.gpu

TEMPS = [0.7, 1.3, 1e-3, 1e-10, 0.0, 1.0, 2.0, 0.5, 0.25, 3.0, 0.1, 1.9999999,
         1.0000001, 0.99999994, 1.5, 0.3, 7.0, 1e-7, 123.456]


def _all_floats(chunk_bits=28):
    n = 1 << chunk_bits
    for c in range(1 << (32 - chunk_bits)):
        yield torch.arange(c * n, (c + 1) * n, dtype=torch.int64, device="cuda") \
            .to(torch.int32).view(torch.float32)


@pytest.mark.parametrize("temp", TEMPS)
def test_quotient_is_ieee_division_for_every_float(temp):
    lib = drs()
    te = max(np.float32(temp), np.float32(1e-10))
    bad = 0
    examples = []
    for x in _all_floats():
        out = torch.empty_like(x)
        lib.drs_scaled_logits(x, float(temp), out)
        ref = x / torch.full_like(x, float(te))      # tensor / tensor: IEEE division
        nan = torch.isnan(out) & torch.isnan(ref)
        diff = (out.view(torch.int32) != ref.view(torch.int32)) & ~nan
        n = int(diff.sum())
        if n:
            bad += n
            idx = diff.nonzero().flatten()[:3]
            examples += [(float(x[i]), float(out[i]), float(ref[i])) for i in idx]
    torch.cuda.synchronize()
    assert bad == 0, f"T={temp}: {bad} quotients differ, e.g. {examples[:3]}"
