"""drs_row_stats_noalloc: the row statistics for callers that cannot
allocate device memory for the library (plugin interfaces that receive only
input and output buffers, or code that must not call cudaMalloc). It keeps
its kernels' records in a fixed device array of the library, and runs calls
whose rows need more in batches of rows.

The test calls it through the C ABI twice in a row (the second call reuses
the array the first one left behind) and compares every output with
drs_row_stats on the same inputs, within the parity tolerances. It is
collected last (file name), runs alone in a fresh process as well as after
the other tests.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import drs
from parity import ENTROPY_ABS

pytestmark = pytest.mark.gpu


def _outputs(rows, vocab, probs):
    dev = "cuda"
    return (torch.full((rows,), -1, dtype=torch.int64, device=dev),
            torch.full((rows,), -1, dtype=torch.int64, device=dev),
            torch.full((rows,), float("nan"), dtype=torch.float32, device=dev),
            torch.zeros(rows, vocab, dtype=torch.bfloat16, device=dev) if probs else None)


def _cases():
    w = workloads.make("tiny")
    yield "tiny", w["logits"].cuda(), w["temps"].cuda(), w["canvas_len"]
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((40, 131072)) * 3).astype(np.float32)   # 22 + 16 tiles per row
    x[5] = -np.inf
    x[5, 70000] = 1.0
    t = torch.tensor([0.0, 0.8, 1.0, 1e-3, 1.4], dtype=torch.float32, device="cuda")
    yield "shared rows", torch.as_tensor(x).cuda(), t, 8
    # more rows than one batch of the fixed array holds (at most 137 rows of
    # 262144 columns): the call runs in batches, row0 and the outputs offset
    g = torch.Generator(device="cuda").manual_seed(4)
    xb = 3.0 * torch.randn(300, 262144, generator=g, device="cuda")
    tb = torch.tensor([0.9, 0.0, 1.2], dtype=torch.float32, device="cuda")
    yield "batched rows", xb, tb, 100


@pytest.mark.parametrize("with_probs", [True, False])
def test_noalloc_matches_row_stats_on_two_calls_in_a_row(with_probs):
    lib = drs()
    code = lib.DRS_PROBS_BF16 if with_probs else lib.DRS_PROBS_NONE
    for name, x, temps, canvas in _cases():
        rows, vocab = x.shape
        ref = lib.row_stats(x, temps, canvas, 77, torch.bfloat16 if with_probs else None)
        for call in range(2):
            a, s, e, p = _outputs(rows, vocab, with_probs)
            lib.drs_row_stats_noalloc(x, temps, canvas, 77, a, s, e, code, p)
            torch.cuda.synchronize()
            assert lib.drs_get_device_error() == 0
            where = f"{name}, call {call + 1}"
            assert torch.equal(a, ref[0]), where
            assert torch.equal(s, ref[1]), where
            assert float((e - ref[2]).abs().max()) <= ENTROPY_ABS, where
            if with_probs:
                d = (p.view(torch.int16).int() - ref[3].view(torch.int16).int()).abs()
                assert int(d.max()) <= 1, where
