"""GPU parity of drs_row_stats_topk: the row statistics and the top-k
logprobs of converged rows from one read of the logits.

Every output is compared with the CPU oracle (row statistics, and top-k
from a sort of each row), and at full size with the two separate calls
(drs_row_stats then drs_topk_logprobs). Rows of unconverged slots keep their
sentinel top-k outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import THREADS, drs, oracle_rows, sample_rows, subset
from parity import ENTROPY_ABS, LOGPROB_ABS, check_row_stats, check_topk

pytestmark = pytest.mark.gpu

SENTINEL_ID = -123456789
SENTINEL_LP = np.float32(-7.25)
BF16 = 1


def _fused(logits_dev, temps, canvas_len, seed, keep, k, probs_dtype=BF16, row0=0):
    lib = drs()
    rows = logits_dev.shape[0]
    ids = torch.full((rows, k), SENTINEL_ID, dtype=torch.int32, device="cuda")
    lps = torch.full((rows, k), float(SENTINEL_LP), dtype=torch.float32, device="cuda")
    pd = {0: None, 1: torch.bfloat16, 2: torch.float16}[probs_dtype]
    a, s, e, p, ids, lps = lib.row_stats_topk(logits_dev, torch.as_tensor(temps).cuda(), canvas_len,
                                              seed, torch.as_tensor(keep).cuda(), k, pd, ids, lps,
                                              row0=row0)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    out = {"argmax": a.cpu().numpy(), "sample": s.cpu().numpy(), "entropy": e.cpu().numpy(),
           "probs": None if p is None else p.view(torch.int16).cpu().numpy().view(np.uint16)}
    return out, ids.cpu().numpy(), lps.cpu().numpy()


def _check(logits_dev, temps, canvas_len, seed, keep, k, rows_sel=None, probs_dtype=BF16,
           row0=0, where=""):
    rows = logits_dev.shape[0]
    g, ids, lps = _fused(logits_dev, temps, canvas_len, seed, keep, k, probs_dtype, row0)
    sel = np.arange(rows) if rows_sel is None else np.asarray(rows_sel, np.int64)
    ref = oracle_rows(logits_dev, temps, canvas_len, seed, probs_dtype, sel, row0=row0)
    near = check_row_stats(subset(g, sel), ref, probs_dtype, where)
    kept = np.asarray(keep)[(np.arange(rows) + row0) // canvas_len] != 0
    assert np.all(ids[~kept] == SENTINEL_ID) and np.all(lps[~kept] == SENTINEL_LP), where
    ksel = sel[kept[sel]]
    if ksel.size:
        x = np.ascontiguousarray(logits_dev[torch.as_tensor(ksel).cuda()].cpu().numpy())
        t = np.asarray(temps, np.float32)[(ksel + row0) // canvas_len]
        ri, rl = oracle.topk_rows(x, t, k, threads=THREADS)
        check_topk(ids[ksel], lps[ksel], ri, rl, where)
    return near


@pytest.mark.parametrize("seed", [0, 2**63 + 7])
def test_tiny_every_row(seed):
    w = workloads.make("tiny")
    near = _check(w["logits"].cuda(), w["temps"].numpy(), 16, seed,
                  np.array([0, 1, 1, 0], np.uint8), 8, where=f"tiny seed {seed}")
    assert near <= 2


@pytest.mark.parametrize("k", [1, 8, 20, 64, 65])
def test_hard_and_easy_rows(k):
    """Normal rows, rows whose candidates overflow (constant, heavy ties),
    rows without a threshold (one-hot, mostly -inf), tiny temperatures."""
    rng = np.random.default_rng(k)
    rows, vocab, canvas = 16, 70001, 2
    x = (rng.standard_normal((rows, vocab)) * 3).astype(np.float32)
    x[0] = 0.25                                      # constant
    x[1] = np.round(x[1])                            # heavy ties
    x[2] = -np.inf
    x[2, 12345] = 1.0                                # one-hot
    x[3][rng.random(vocab) < 0.999] = -np.inf        # a few finite values
    x[4, ::1000] = 30.0                              # many equal maxima
    x[5, 70000] = 50.0                               # max in the last column
    temps = np.array([1.0, 0.7, 0.0, 1e-3, 1.3, 1e-10, 2.0, 0.5], np.float32)
    keep = np.array([1, 1, 1, 0, 1, 1, 0, 1], np.uint8)
    _check(torch.as_tensor(x).cuda(), temps, canvas, 17, keep, k, where=f"k={k}")


def test_row_offset_split_matches_one_call():
    """keep and temps are indexed by global slot: two calls on the halves of
    a batch (row0 = 0 and row0 = rows/2) equal one call."""
    w = workloads.make("tiny")
    x = w["logits"].cuda()
    temps, keep = w["temps"].numpy(), np.array([1, 0, 1, 1], np.uint8)
    whole = _fused(x, temps, 16, 5, keep, 8)
    lo = _fused(x[:32], temps, 16, 5, keep, 8, row0=0)
    hi = _fused(x[32:], temps, 16, 5, keep, 8, row0=32)
    for key in ("argmax", "sample", "entropy", "probs"):
        assert np.array_equal(whole[0][key], np.concatenate([lo[0][key], hi[0][key]])), key
    assert np.array_equal(whole[1], np.concatenate([lo[1], hi[1]]))
    assert np.array_equal(whole[2], np.concatenate([lo[2], hi[2]]))


def test_empty_and_k_zero():
    lib = drs()
    x = torch.zeros(0, 16, device="cuda")
    out = lib.row_stats_topk(x, torch.ones(1, device="cuda"), 1, 0,
                             torch.ones(1, dtype=torch.uint8, device="cuda"), 4)
    assert out[0].numel() == 0
    w = workloads.make("tiny")
    g, ids, lps = _fused(w["logits"].cuda(), w["temps"].numpy(), 16, 3, np.ones(4, np.uint8), 0)
    ref = oracle_rows(w["logits"], w["temps"].numpy(), 16, 3, BF16, np.arange(64))
    check_row_stats(g, ref, BF16, "k = 0")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["step", "adversarial"])
def test_full_size_equals_separate_calls_and_oracle(name):
    """The bench's launch: the whole workload in one call. Equal to
    drs_row_stats + drs_topk_logprobs on the same inputs (integers exactly,
    floating point within the parity tolerances); sampled rows against the
    oracle."""
    lib = drs()
    w = workloads.make(name, device="cuda")
    V, k, cl = w["vocab"], w["k"], w["canvas_len"]
    x = w["logits"][:, :V]
    temps = w["temps"].cuda()
    keep = w["keep"].cuda()
    pd = {0: None, 1: torch.bfloat16, 2: torch.float16}[w["probs_dtype"]]
    a, s, e, p, ids, lps = lib.row_stats_topk(x, temps, cl, 0, keep, k, pd)
    a2, s2, e2, p2 = lib.row_stats(x, temps, cl, 0, pd)
    ids2, lps2 = lib.topk_logprobs(x, temps, cl, keep, k)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    # the two paths may split a row over a different number of CTAs, so
    # sums can round differently: integers exactly, the rest within the
    # parity tolerances
    assert torch.equal(a, a2) and torch.equal(s, s2)
    assert float((e - e2).abs().max()) <= ENTROPY_ABS
    if p is not None:
        d = (p.view(torch.int16).int() - p2.view(torch.int16).int()).abs()
        assert int(d.max()) <= 1
    assert torch.equal(ids, ids2)
    both_nan = lps.isnan() & lps2.isnan()
    close = (lps - lps2).abs() <= torch.maximum(torch.full_like(lps, LOGPROB_ABS),
                                                 lps2.abs() * 2.0**-23)
    assert bool((both_nan | close | (lps == lps2)).all())
    sel = sample_rows(w["rows"], 12, seed=3, always=(0, 1, w["rows"] - 1))
    g = {"argmax": a.cpu().numpy(), "sample": s.cpu().numpy(), "entropy": e.cpu().numpy(),
         "probs": None if p is None else p.view(torch.int16).cpu().numpy().view(np.uint16)}
    temps_h = w["temps"].cpu().numpy()
    ref = oracle_rows(x, temps_h, cl, 0, w["probs_dtype"], sel)
    check_row_stats(subset(g, sel), ref, w["probs_dtype"], name)
    kept = w["keep"].cpu().numpy()[sel // cl] != 0
    ksel = sel[kept]
    xs = np.ascontiguousarray(x[torch.as_tensor(ksel).cuda()].cpu().numpy())
    ri, rl = oracle.topk_rows(xs, temps_h[ksel // cl], k, threads=THREADS)
    check_topk(ids.cpu().numpy()[ksel], lps.cpu().numpy()[ksel], ri, rl, name)
