"""GPU parity on rows longer than 524288 columns, up to DRS_MAX_VOCAB (2^21).

These rows go through the two streaming passes in up to 256 tiles of 8192
columns, merged by the merge's long-row instantiation. Their exact top-k
comes from one CTA per row reading the row five times, because a team of
CTAs cannot stage them. That path takes the rows the passes leave (no
threshold, too many candidates) and every kept row when k > 64. Each case
mixes normal rows with the hard ones: constant, one-hot, heavy ties, a few
finite values, and many equal maxima.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import THREADS, drs, oracle_rows, subset
from parity import check_row_stats, check_topk

pytestmark = pytest.mark.gpu

SENTINEL_ID = -123456789
SENTINEL_LP = np.float32(-7.25)
BF16 = 1


def _rows(vocab, seed, rows=8):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, vocab)) * 3).astype(np.float32)
    x[0] = 0.25                                      # constant: the k lowest columns
    x[1] = np.round(x[1])                            # heavy ties
    x[2] = -np.inf
    x[2, vocab - 7] = 1.0                            # one-hot near the end
    x[3][rng.random(vocab) < 0.9999] = -np.inf       # a few finite values
    x[4, ::5000] = 30.0                              # many equal maxima
    x[5, vocab - 1] = 50.0                           # max in the last column
    return x


def _topk_check(x, temps, canvas, keep, k, where):
    lib = drs()
    rows = x.shape[0]
    dev = torch.as_tensor(x).cuda()
    ids = torch.full((rows, k), SENTINEL_ID, dtype=torch.int32, device="cuda")
    lps = torch.full((rows, k), float(SENTINEL_LP), dtype=torch.float32, device="cuda")
    lib.topk_logprobs(dev, torch.as_tensor(temps).cuda(), canvas, torch.as_tensor(keep).cuda(), k,
                      ids, lps)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    ids, lps = ids.cpu().numpy(), lps.cpu().numpy()
    kept = np.repeat(keep != 0, canvas)[:rows]
    assert np.all(ids[~kept] == SENTINEL_ID) and np.all(lps[~kept] == SENTINEL_LP), where
    sel = np.flatnonzero(kept)
    ri, rl = oracle.topk_rows(np.ascontiguousarray(x[sel]), temps[sel // canvas], k, threads=THREADS)
    check_topk(ids[sel], lps[sel], ri, rl, where)


@pytest.mark.parametrize("vocab,k", [(600000, 8), (600000, 100), (1048576, 64), (1048576, 1024),
                                     (2097152, 20)])
def test_topk_logprobs_long_rows(vocab, k):
    x = _rows(vocab, vocab + k)
    temps = np.array([1.0, 0.7, 1e-3, 1.3], np.float32)
    keep = np.array([1, 1, 1, 0], np.uint8)
    _topk_check(x, temps, 2, keep, k, f"V={vocab} k={k}")


@pytest.mark.parametrize("vocab", [1048576, 2097152])
def test_row_stats_topk_long_rows(vocab):
    """drs_row_stats_topk: statistics, probabilities and top-20 of the kept
    rows against the oracle; the hard rows' top-k by the one-CTA kernel."""
    lib = drs()
    x = _rows(vocab, 3)
    rows, canvas, k = x.shape[0], 2, 20
    temps = np.array([1.0, 0.7, 0.0, 1.3], np.float32)
    keep = np.array([1, 1, 1, 0], np.uint8)
    dev = torch.as_tensor(x).cuda()
    ids = torch.full((rows, k), SENTINEL_ID, dtype=torch.int32, device="cuda")
    lps = torch.full((rows, k), float(SENTINEL_LP), dtype=torch.float32, device="cuda")
    a, s, e, p, ids, lps = lib.row_stats_topk(dev, torch.as_tensor(temps).cuda(), canvas, 29,
                                              torch.as_tensor(keep).cuda(), k, torch.bfloat16, ids, lps)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    g = {"argmax": a.cpu().numpy(), "sample": s.cpu().numpy(), "entropy": e.cpu().numpy(),
         "probs": p.view(torch.int16).cpu().numpy().view(np.uint16)}
    sel = np.arange(rows)
    ref = oracle_rows(dev, temps, canvas, 29, BF16, sel)
    check_row_stats(subset(g, sel), ref, BF16, f"V={vocab}")
    ids, lps = ids.cpu().numpy(), lps.cpu().numpy()
    kept = np.repeat(keep != 0, canvas)
    assert np.all(ids[~kept] == SENTINEL_ID) and np.all(lps[~kept] == SENTINEL_LP)
    ksel = np.flatnonzero(kept)
    ri, rl = oracle.topk_rows(np.ascontiguousarray(x[ksel]), temps[ksel // canvas], k, threads=THREADS)
    check_topk(ids[ksel], lps[ksel], ri, rl, f"V={vocab} top-k")
