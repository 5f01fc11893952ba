"""GPU parity of drs_row_stats_seeds: several noise seeds in one call.

The argmax equals drs_row_stats's and the sample of seed s equals
drs_row_stats with that seed, bit for bit (every implementation scores the
race's survivors exactly: s = x / Te by the exact quotient plus the fp32
noise); the entropy and the probabilities agree within the parity
tolerances (one-seed calls may take the one-read cluster kernel, several
seeds the two passes, whose roundings of the exponent differ), and all of
them match the oracle on sampled rows. The strided workload is the multi-seed configuration of the
task (eight seeds, no probabilities, T = 1).
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import drs, oracle_rows, sample_rows, subset
from parity import ENTROPY_ABS, check_row_stats

pytestmark = pytest.mark.gpu

SEEDS = [0, 1, 7, 2**63 + 5, 12345, 2**32 - 1, 2**32, 99]


def _compare_to_single(x, temps, canvas, seeds, probs_dtype, row0=0):
    lib = drs()
    a, smp, e, p = lib.row_stats_seeds(x, temps, canvas, seeds, probs_dtype, row0=row0)
    for i, sd in enumerate(seeds):
        a1, s1, e1, p1 = lib.row_stats(x, temps, canvas, sd, probs_dtype, row0=row0)
        torch.cuda.synchronize()
        assert torch.equal(a, a1)
        assert torch.equal(smp[i], s1), f"seed {sd}"
        assert float((e - e1).abs().max()) <= ENTROPY_ABS if e.numel() else True
        if p is not None:
            c, c1 = p.view(torch.int16).int(), p1.view(torch.int16).int()
            assert int((c - c1).abs().max()) <= 1
    assert lib.drs_get_device_error() == 0
    return a, smp, e, p


@pytest.mark.parametrize("n", [1, 3, 8])
def test_tiny_every_row_equals_single_seed_calls(n):
    w = workloads.make("tiny")
    x, t = w["logits"].cuda(), w["temps"].cuda()
    a, smp, e, p = _compare_to_single(x, t, 16, SEEDS[:n], torch.bfloat16)
    for i in range(n):
        g = {"argmax": a.cpu().numpy(), "sample": smp[i].cpu().numpy(),
             "entropy": e.cpu().numpy(),
             "probs": p.view(torch.int16).cpu().numpy().view(np.uint16)}
        ref = oracle_rows(w["logits"], w["temps"].numpy(), 16, SEEDS[i], 1, np.arange(64))
        assert check_row_stats(g, ref, 1, f"seed {SEEDS[i]}") <= 2


def test_special_rows_and_row0():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((24, 70001)) * 3).astype(np.float32)
    x[0] = -np.inf
    x[1] = 0.5
    x[2] = -np.inf
    x[2, 50000] = 2.0
    t = torch.tensor([0.0, 1.0, 1e-3, 1.7], dtype=torch.float32, device="cuda")
    _compare_to_single(torch.as_tensor(x).cuda(), t, 4, SEEDS[:5], None, row0=8)


def test_argument_errors():
    lib = drs()
    x = torch.zeros(4, 64, device="cuda")
    t = torch.ones(1, device="cuda")
    with pytest.raises(lib.DrsError):
        lib.row_stats_seeds(x, t, 4, list(range(9)))
    assert lib.drs_row_stats_seeds_workspace_bytes(4, 64, 0) == 0
    assert lib.drs_row_stats_seeds_workspace_bytes(4, 64, 9) == 0


@pytest.mark.slow
def test_strided_workload_eight_seeds():
    """The strided workload (2048 x 262144 inside a padded stride, T = 1, no
    probabilities) with its eight seeds in one call; sampled rows against the
    oracle."""
    lib = drs()
    w = workloads.make("strided", device="cuda")
    V = w["vocab"]
    x = w["logits"][:, :V]
    temps = w["temps"].cuda()
    seeds = list(range(8))
    a, smp, e, _ = lib.row_stats_seeds(x, temps, w["canvas_len"], seeds, None)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    sel = sample_rows(w["rows"], 6, seed=5, always=(0, w["rows"] - 1))
    for i, sd in enumerate(seeds):
        g = {"argmax": a.cpu().numpy(), "sample": smp[i].cpu().numpy(),
             "entropy": e.cpu().numpy(), "probs": None}
        ref = oracle_rows(x, w["temps"].cpu().numpy(), w["canvas_len"], sd, 0, sel)
        check_row_stats(subset(g, sel), ref, 0, f"strided seed {sd}")


@pytest.mark.parametrize("vocab", [600000, 2097152])
def test_long_rows_equal_single_seed_calls(vocab):
    """Rows long enough that the merge shares each row among the warps of a
    CTA: every seed's sample equals a single-seed call's, and each seed's
    statistics equal the oracle's on every row."""
    rng = np.random.default_rng(vocab)
    x = (rng.standard_normal((6, vocab)) * 3).astype(np.float32)
    x[1] = 0.5                                  # constant
    x[2, vocab - 1] = 40.0                      # the max in the last column
    x[3][rng.random(vocab) < 0.999] = -np.inf   # a few finite values
    temps = np.array([1.0, 0.6, 1.4], np.float32)
    dev = torch.as_tensor(x).cuda()
    seeds = SEEDS[:3]
    a, smp, e, p = _compare_to_single(dev, torch.as_tensor(temps).cuda(), 2, seeds, torch.bfloat16)
    sel = np.arange(x.shape[0])
    for i, sd in enumerate(seeds):
        g = {"argmax": a.cpu().numpy(), "sample": smp[i].cpu().numpy(),
             "entropy": e.cpu().numpy(),
             "probs": p.view(torch.int16).cpu().numpy().view(np.uint16)}
        ref = oracle_rows(dev, temps, 2, sd, 1, sel)
        assert check_row_stats(g, ref, 1, f"V={vocab} seed {sd}") <= 1
