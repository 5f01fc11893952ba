"""GPU parity of drs_topk_logprobs against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import THREADS, drs, sample_rows
from parity import check_topk

pytestmark = pytest.mark.gpu

SENTINEL_ID = -123456789
SENTINEL_LP = np.float32(-7.25)


def _run(logits_dev, temps, canvas_len, keep, k):
    lib = drs()
    rows = logits_dev.shape[0]
    ids = torch.full((rows, k), SENTINEL_ID, dtype=torch.int32, device="cuda")
    lps = torch.full((rows, k), float(SENTINEL_LP), dtype=torch.float32, device="cuda")
    lib.topk_logprobs(logits_dev, torch.as_tensor(temps).cuda(), canvas_len,
                      torch.as_tensor(keep).cuda(), k, ids, lps)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    return ids.cpu().numpy(), lps.cpu().numpy()


def _check(logits_dev, temps, canvas_len, keep, k, rows_sel=None, where=""):
    rows = logits_dev.shape[0]
    ids, lps = _run(logits_dev, temps, canvas_len, keep, k)
    kept = np.repeat(np.asarray(keep) != 0, canvas_len)[:rows]
    # rows of slots that are not kept are never written
    assert np.all(ids[~kept] == SENTINEL_ID) and np.all(lps[~kept] == SENTINEL_LP), where
    sel = np.flatnonzero(kept) if rows_sel is None else np.asarray(
        [r for r in rows_sel if kept[r]], dtype=np.int64)
    if sel.size == 0:
        return
    x = np.ascontiguousarray(logits_dev[torch.as_tensor(sel).cuda()].cpu().numpy())
    t = np.asarray(temps, np.float32)[sel // canvas_len]
    ri, rl = oracle.topk_rows(x, t, k, threads=THREADS)
    check_topk(ids[sel], lps[sel], ri, rl, where)


def test_tiny_workload_all_and_masked():
    w = workloads.make("tiny")
    x = w["logits"].cuda()
    _check(x, w["temps"].numpy(), 16, np.ones(4, np.uint8), 8, where="tiny all kept")
    _check(x, w["temps"].numpy(), 16, np.array([0, 1, 0, 1], np.uint8), 8, where="tiny masked")
    _check(x, w["temps"].numpy(), 16, np.zeros(4, np.uint8), 8, where="tiny none kept")


@pytest.mark.parametrize("vocab,k", [(1, 1), (5, 5), (7, 3), (100, 100), (4097, 64),
                                     (16385, 20), (40003, 64), (131072, 64), (70001, 1024),
                                     (9000, 600)])
def test_shapes_ties_and_masks(vocab, k):
    rows, canvas = 8, 2
    rng = np.random.default_rng(vocab + k)
    x = (rng.standard_normal((rows, vocab)) * 2).astype(np.float32)
    x[rng.random((rows, vocab)) < 0.3] = -np.inf
    x[0] = 0.5                                           # constant: the k lowest columns
    x[1] = -np.inf
    x[1, vocab // 2] = 0.0                               # one-hot, then -inf by column
    x[2] = np.round(x[2] * 2) / 2                        # heavy ties
    if vocab >= 8:
        x[3, 1], x[3, 6] = -0.0, 0.0                     # signed zeros tie
        x[3, :][x[3, :] > 0] = -1.0
    temps = np.array([0.0, 1e-3, 1.0, 0.7], np.float32)
    keep = np.array([1, 1, 0, 1], np.uint8)
    for pad in (0, 3):
        buf = np.full((rows, vocab + pad), np.nan, np.float32)
        buf[:, :vocab] = x
        dev = torch.as_tensor(buf).cuda()[:, :vocab]
        _check(dev, temps, canvas, keep, k, where=f"V={vocab} k={k} pad={pad}")


def test_all_neg_inf_row_gives_nan_logprobs():
    x = np.full((1, 1000), -np.inf, np.float32)
    ids, lps = _run(torch.as_tensor(x).cuda(), np.array([1.0], np.float32), 1,
                    np.ones(1, np.uint8), 4)
    assert list(ids[0]) == [0, 1, 2, 3] and np.all(np.isnan(lps[0]))


def test_k_zero_is_a_no_op():
    x = torch.randn(4, 64, device="cuda")
    ids, lps = _run(x, np.ones(4, np.float32), 1, np.ones(4, np.uint8), 0)
    assert ids.shape == (4, 0)


# ------------------------------------------------------------- full sizes

def _full(name, n_sample):
    w = workloads.make(name, device="cuda")
    V = w["vocab"]
    view = w["logits"][:, :V]
    sel = sample_rows(w["rows"], n_sample, seed=2)
    _check(view, w["temps"].cpu().numpy(), w["canvas_len"], w["keep"].cpu().numpy(), w["k"],
           rows_sel=sel, where=name)
    del w, view
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_adversarial_workload_topk():
    _full("adversarial", 96)


@pytest.mark.slow
def test_step_workload_topk():
    _full("step", 24)


@pytest.mark.slow
def test_large_workload_topk():
    _full("large", 12)
