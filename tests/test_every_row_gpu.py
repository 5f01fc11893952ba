"""Every row of each full-size workload against the oracle.

Each workload runs the way the bench launches it: the whole batch in one
call (drs_row_stats_topk with the workload's keep mask and k; the strided
batch through drs_row_stats_seeds with its eight seeds). Then every row is
compared with the oracle: argmax, sample (for each seed), entropy,
probabilities, and the top-k ids and logprobs of every row of a converged
slot. The oracle works through the rows in chunks on the host's cores, so
host memory stays at a few hundred MB per chunk.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import THREADS, drs
from parity import check_row_stats, check_topk

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TORCH_PD = {0: None, 1: torch.bfloat16, 2: torch.float16}
CHUNK = 512


def _host(t):
    return t.cpu().numpy()


def _codes(p):
    return None if p is None else p.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["tiny", "step", "adversarial", "large"])
def test_every_row_of_the_fused_call(name):
    lib = drs()
    w = workloads.make(name, device="cuda")
    rows, V, k, cl, pd = w["rows"], w["vocab"], w["k"], w["canvas_len"], w["probs_dtype"]
    x = w["logits"][:, :V]
    temps_h = w["temps"].cpu().numpy()
    keep_h = w["keep"].cpu().numpy()
    a, s, e, p, ids, lps = lib.row_stats_topk(x, w["temps"].cuda(), cl, 0, w["keep"].cuda(), k,
                                              TORCH_PD[pd])
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    a, s, e, ids, lps = _host(a), _host(s), _host(e), _host(ids), _host(lps)
    near = 0
    for r0 in range(0, rows, CHUNK):
        r1 = min(rows, r0 + CHUNK)
        gids = np.arange(r0, r1, dtype=np.int64)
        xs = np.ascontiguousarray(x[r0:r1].cpu().numpy())
        ref = oracle.row_stats_rows(xs, gids, temps_h[gids // cl], 0, pd, threads=THREADS)
        got = {"argmax": a[r0:r1], "sample": s[r0:r1], "entropy": e[r0:r1],
               "probs": None if p is None else _codes(p[r0:r1])}
        near += check_row_stats(got, ref, pd, f"{name} rows {r0}..{r1}")
        kept = np.flatnonzero(keep_h[gids // cl] != 0)
        if k and kept.size:
            ri, rl = oracle.topk_rows(np.ascontiguousarray(xs[kept]), temps_h[gids[kept] // cl], k,
                                      threads=THREADS)
            check_topk(ids[r0 + kept], lps[r0 + kept], ri, rl, f"{name} top-k rows {r0}..{r1}")
        # rows of unconverged slots keep the caller's fill
        skipped = r0 + np.flatnonzero(keep_h[gids // cl] == 0)
        if k and skipped.size:
            assert (ids[skipped] == -1).all() and np.isnan(lps[skipped]).all()
        del xs, ref
    # near ties are counted, not failed (at T = 1e-3 and 1e-10 an fp32 score
    # of |s| up to 1e10 has an ulp far above the noise, so the adversarial
    # recipe's rows of equal maxima tie in fp32)
    print(f"{name}: {near} near-tie sample mismatches of {rows} rows")


def test_every_row_of_the_strided_seeds_call():
    lib = drs()
    w = workloads.make("strided", device="cuda")
    rows, V, cl, pd = w["rows"], w["vocab"], w["canvas_len"], w["probs_dtype"]
    seeds = list(w["seeds"])
    x = w["logits"][:, :V]
    assert x.stride(0) > V
    temps_h = w["temps"].cpu().numpy()
    a, smp, e, p = lib.row_stats_seeds(x, w["temps"].cuda(), cl, seeds, TORCH_PD[pd])
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    a, smp, e = _host(a), _host(smp), _host(e)
    near = 0
    for r0 in range(0, rows, CHUNK):
        r1 = min(rows, r0 + CHUNK)
        gids = np.arange(r0, r1, dtype=np.int64)
        xs = np.ascontiguousarray(x[r0:r1].cpu().numpy())
        for i, sd in enumerate(seeds):
            ref = oracle.row_stats_rows(xs, gids, temps_h[gids // cl], sd,
                                        pd if i == 0 else 0, threads=THREADS)
            got = {"argmax": a[r0:r1], "sample": smp[i, r0:r1], "entropy": e[r0:r1],
                   "probs": None if (p is None or i) else _codes(p[r0:r1])}
            near += check_row_stats(got, ref, pd if i == 0 else 0,
                                    f"strided seed {sd} rows {r0}..{r1}")
        del xs
    print(f"strided: {near} near-tie sample mismatches of {rows * len(seeds)} samples")


@pytest.mark.parametrize("name", ["step", "adversarial"])
def test_repeated_full_size_calls_are_bit_identical(name):
    """A call divides its rows between the cluster kernel and the two passes,
    which sum a row's exponentials in different orders; the division must be
    the same on every run, so repeated calls give the same bits."""
    lib = drs()
    w = workloads.make(name, device="cuda")
    V, k, cl, pd = w["vocab"], w["k"], w["canvas_len"], w["probs_dtype"]
    x = w["logits"][:, :V]
    temps, keep = w["temps"].cuda(), w["keep"].cuda()
    first = lib.row_stats_topk(x, temps, cl, 0, keep, k, TORCH_PD[pd])
    for _ in range(4):
        again = lib.row_stats_topk(x, temps, cl, 0, keep, k, TORCH_PD[pd])
        torch.cuda.synchronize()
        for a, b in zip(first, again):
            if a is None:
                continue
            if a.is_floating_point():
                a, b = a.view(torch.int16 if a.element_size() == 2 else torch.int32), \
                    b.view(torch.int16 if b.element_size() == 2 else torch.int32)
            assert torch.equal(a, b)
    # the top-k-only call and the stash's rows too
    ids1, lp1 = lib.topk_logprobs(x, temps, cl, keep, k)
    ids2, lp2 = lib.topk_logprobs(x, temps, cl, keep, k)
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids2)
    assert torch.equal(lp1.view(torch.int32), lp2.view(torch.int32))


def test_large_batch_is_the_same_bytes_on_every_draw():
    """The large recipe's mixture columns may repeat within a row; the batch
    must still be reproducible, or runs could not be compared."""
    a = workloads.make_logits("large", device="cuda", rows=256)
    b = workloads.make_logits("large", device="cuda", rows=256)
    assert torch.equal(a, b)
