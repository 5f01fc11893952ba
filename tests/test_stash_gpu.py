"""GPU parity of drs_stash_converged_logprobs against the oracle's stash.

Requests with permuted src and slots, a mix of keep flags and valid
lengths, temperatures 0, 1e-3 and ordinary ones, rows that are constant,
tied, -inf everywhere, or mostly -inf. Both paths are covered: the
request's token ids (counts 0 to 4, one id outside the vocabulary) and the
num_topk largest. Values are logprobs or the scaled logits themselves.
Stash rows the call must not write are filled with a sentinel first and
checked bit for bit. Ids are exact; logprobs are within the parity
tolerance; scaled logits are exact.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import drs
from parity import check_topk

pytestmark = pytest.mark.gpu

SENT_ID, SENT_V, SENT_R = -123456789, np.float32(-7.25), -55


def _batch(seed, vocab, m=5, canvas=4):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((m * canvas + 3, vocab)) * 2).astype(np.float32)
    x[rng.random(x.shape) < 0.2] = -np.inf
    x[3] = np.round(x[3])                         # ties
    x[5] = 0.5                                    # constant
    x[6] = -np.inf                                # all -inf
    x[9][rng.random(vocab) < 0.999] = -np.inf     # a few finite values
    src = rng.permutation(m).astype(np.int32)
    slots = rng.permutation(m + 2)[:m].astype(np.int32)
    keep = np.array([1, 0, 1, 1, 1], np.uint8)
    valid = np.array([4, 4, 2, 0, 3], np.int32)
    temps = np.array([1.0, 0.7, 0.0, 1e-3, 1.3], np.float32)
    tok = np.array([[5, vocab - 1, 0, 17], [1, 2, 3, 4], [9, 9, vocab, 2], [0, 0, 0, 0],
                    [42 % vocab, 7, 7, 1]], np.int32)
    nti = np.array([4, 2, 4, 1, 0], np.int32)
    return x, src, slots, keep, valid, temps, tok, nti, m, canvas


def _run(x, canvas, src, slots, keep, valid, temps, k, nti, tok, out_slots, width, mode):
    lib = drs()
    dev = lambda a: torch.as_tensor(a).cuda()
    ids = torch.full((out_slots, canvas, width), SENT_ID, dtype=torch.int32, device="cuda")
    vals = torch.full((out_slots, canvas, width), float(SENT_V), dtype=torch.float32, device="cuda")
    ranks = torch.full((out_slots, canvas), SENT_R, dtype=torch.int32, device="cuda")
    lib.stash_converged_logprobs(dev(x), canvas, dev(src), dev(slots), dev(keep), dev(valid),
                                 dev(temps), k, None if nti is None else dev(nti),
                                 None if tok is None else dev(tok), ids, vals, ranks,
                                 logits_mode=mode)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    return ids.cpu().numpy(), vals.cpu().numpy(), ranks.cpu().numpy()


def _compare(x, canvas, src, slots, keep, valid, temps, k, nti, tok, width, mode, where):
    out_slots = len(src) + 2
    g_ids, g_vals, g_ranks = _run(x, canvas, src, slots, keep, valid, temps, k, nti, tok,
                                  out_slots, width, mode)
    r_ids, r_vals, r_ranks = oracle.stash(x, canvas, src, slots, keep, valid, temps, k, nti, tok,
                                          out_slots, width, logits_mode=mode)
    written = r_ranks != -1
    assert np.all(g_ids[~written] == SENT_ID) and np.all(g_vals[~written] == SENT_V), where
    assert np.all(g_ranks[~written] == SENT_R), where
    assert np.array_equal(g_ranks[written], r_ranks[written]), where
    gi, gv = g_ids[written], g_vals[written]
    ri, rv = r_ids[written], r_vals[written]
    if mode:
        assert np.array_equal(gi, ri), where
        same = (gv == rv.astype(np.float32)) | (np.isnan(gv) & np.isnan(rv))
        assert same.all(), f"{where}: scaled logits differ at {np.argwhere(~same)[:3]}"
    else:
        check_topk(gi, gv, ri, rv, where)


@pytest.mark.parametrize("vocab,k", [(777, 0), (777, 5), (70001, 64), (70001, 100),
                                     (600000, 20)])
@pytest.mark.parametrize("ids_path", [False, True])
@pytest.mark.parametrize("mode", [False, True])
def test_stash_against_oracle(vocab, k, ids_path, mode):
    x, src, slots, keep, valid, temps, tok, nti, m, canvas = _batch(vocab + k, vocab)
    width = k + 3 if not ids_path else max(k + 1, 6)
    _compare(x, canvas, src, slots, keep, valid, temps, k, nti if ids_path else None,
             tok if ids_path else None, width, mode,
             f"V={vocab} k={k} ids={ids_path} logits={mode}")


def test_stash_token_counts_past_the_list():
    """num_token_ids larger than ids_stride: a request's list holds ids_stride
    ids, the rest of the count is padding. The last request's count runs
    past the end of the token-id array, which must not be read."""
    x, src, slots, keep, valid, temps, tok, nti, m, canvas = _batch(4, 5000)
    keep = np.ones(m, np.uint8)
    valid = np.full(m, canvas, np.int32)
    nti = np.array([4, 9, 4, 1, 7], np.int32)
    _compare(x, canvas, src, slots, keep, valid, temps, 2, nti, tok, 12, False, "counts past the list")


def test_stash_width_truncates_token_ids():
    x, src, slots, keep, valid, temps, tok, nti, m, canvas = _batch(3, 5000)
    _compare(x, canvas, src, slots, keep, valid, temps, 2, nti, tok, 3, False, "width 3")


def test_stash_step_sized_batch():
    """8 requests x canvas 256 x 262144 columns, every other request kept,
    top-20: sampled stash rows against the oracle."""
    rng = np.random.default_rng(11)
    m, canvas, vocab, k = 8, 256, 262144, 20
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x_dev = torch.randn(m * canvas, vocab, generator=g, device="cuda") * 3.0
    src = rng.permutation(m).astype(np.int32)
    slots = rng.permutation(m).astype(np.int32)
    keep = (np.arange(m) % 2 == 0).astype(np.uint8)
    valid = np.full(m, canvas, np.int32)
    valid[2] = 100
    temps = (0.5 + rng.random(m)).astype(np.float32)
    lib = drs()
    dev = lambda a: torch.as_tensor(a).cuda()
    ids, vals, ranks = lib.stash_converged_logprobs(x_dev, canvas, dev(src), dev(slots), dev(keep),
                                                    dev(valid), dev(temps), k, width=k + 1)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    ids, vals, ranks = ids.cpu().numpy(), vals.cpu().numpy(), ranks.cpu().numpy()
    for j in np.flatnonzero(keep):
        for pos in rng.choice(valid[j], 3, replace=False):
            row = int(src[j]) * canvas + int(pos)
            x = np.ascontiguousarray(x_dev[row:row + 1].cpu().numpy())
            ri, rl = oracle.topk_rows(x, temps[j:j + 1], k)
            o = (int(slots[j]), int(pos))
            assert ids[o][0] == ri[0, 0] and ranks[o] == 1
            check_topk(ids[o][None, 1:], vals[o][None, 1:], ri, rl, f"request {j} pos {pos}")
    for j in np.flatnonzero(keep == 0):
        assert np.all(ids[slots[j]] == -1) and np.all(ranks[slots[j]] == -1)
    assert np.all(ids[slots[2], 100:] == -1)          # positions past valid[2]


def test_stash_skips_requests_outside_the_buffers():
    """A request whose logits rows lie past the logits, or whose slot lies
    past the stash, is skipped without touching any output; the others are
    those of the oracle run without it."""
    x, src, slots, keep, valid, temps, tok, nti, m, canvas = _batch(21, 999)
    keep = np.ones(m, np.uint8)
    bad_src, bad_slot = src.copy(), slots.copy()
    bad_src[1] = 10**6                      # rows far past the logits
    bad_slot[4] = m + 2                     # one past the stash's slots (valid[4] = 3)
    out_slots, width, k = m + 2, 6, 4
    g_ids, g_vals, g_ranks = _run(x, canvas, bad_src, bad_slot, keep, valid, temps, k, None, None,
                                  out_slots, width, False)
    ok = np.array([j not in (1, 4) for j in range(m)])
    r_ids, r_vals, r_ranks = oracle.stash(x, canvas, src[ok], slots[ok], keep[ok], valid[ok],
                                          temps[ok], k, None, None, out_slots, width)
    written = r_ranks != -1
    assert np.all(g_ids[~written] == SENT_ID) and np.all(g_ranks[~written] == SENT_R)
    assert np.array_equal(g_ranks[written], r_ranks[written])
    check_topk(g_ids[written], g_vals[written], r_ids[written], r_vals[written], "skipped requests")


@pytest.mark.parametrize("vocab", [777, 70001])
def test_topk_values_equal_the_division_path(vocab):
    """In logprobs mode a top-k column takes the top-k's own logprob, a
    token-id column one IEEE division and (s - max) - log S: with one
    position per request and each request's top-k ids passed back as its
    token ids, both paths must give the same bits (the argmax column too)."""
    rng = np.random.default_rng(7)
    m, k = 24, 8
    x = (rng.standard_normal((m, vocab)) * 3).astype(np.float32)
    x[2] = np.round(x[2])                      # ties
    x[4][rng.random(vocab) < 0.999] = -np.inf  # fewer finite values than k
    x[5] = -np.inf                             # all -inf
    src = np.arange(m, dtype=np.int32)
    slots = np.arange(m, dtype=np.int32)
    keep = np.ones(m, np.uint8)
    valid = np.ones(m, np.int32)
    temps = np.array([0.7, 1.0, 1.3, 1e-3, 0.0, 2.0] * (m // 6), np.float32)
    ids1, vals1, _ = _run(x, 1, src, slots, keep, valid, temps, k, None, None, m, k + 1, 0)
    tok = np.ascontiguousarray(ids1[:, 0, 1:]).astype(np.int32)
    nti = np.full(m, k, np.int32)
    ids2, vals2, _ = _run(x, 1, src, slots, keep, valid, temps, k, nti, tok, m, k + 1, 0)
    assert np.array_equal(ids1, ids2)
    same = (vals1.view(np.uint32) == vals2.view(np.uint32)) | (np.isnan(vals1) & np.isnan(vals2))
    assert same.all(), f"values differ at {np.argwhere(~same)[:4]}"
