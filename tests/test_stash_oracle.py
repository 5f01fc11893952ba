"""Pins of the oracle's stash (stash_converged_logprobs on page
"vllm.model_executor.models.diffusion_gemma_sampler", its docstring) to facts
that do not come from the stash code: a worked example in closed form, the
separately written top-k routine, a numpy log-softmax, IEEE fp32 division,
and the layout rules of the docstring (argmax first, then token ids or the
top-k, padding with id 0 at -inf, rows of requests not kept untouched).
CPU only.
"""
import math

import numpy as np
import pytest

import oracle


def _log_softmax(x, temp):
    s = (x / np.float32(max(temp, 1e-10))).astype(np.float32) + np.float32(0.0)
    m = float(np.max(s))
    if m == -np.inf:                              # every column -inf: no log-softmax
        return s, np.full(s.shape, np.nan)
    fin = s[np.isfinite(s)].astype(np.float64)
    return s, s.astype(np.float64) - m - math.log(np.sum(np.exp(fin - m)))


def test_worked_example():
    """Two requests, canvas 2. Request 0 (rows 2-3, slot 0, T = 1) keeps two
    positions; request 1 (rows 0-1, slot 1, T = 0.5) keeps one. The values
    below are the closed forms of the log-softmax of these rows."""
    x = np.array([[1, 3, 3, -np.inf, 0, 2], [0, 0, 0, 0, 0, 0],
                  [5, 4, 3, 2, 1, 0], [-1, -2, -3, -4, -5, -6]], np.float32)
    ids, vals, ranks = oracle.stash(x, 2, [1, 0], [0, 1], [1, 1], [2, 1], [1.0, 0.5], 3, None,
                                    None, 2, 5)
    lse_desc = math.log(sum(math.exp(-k) for k in range(6)))       # rows 2 and 3
    for p in (0, 1):
        assert list(ids[0, p]) == [0, 0, 1, 2, 0]
        np.testing.assert_allclose(vals[0, p, :4], [-lse_desc, -lse_desc, -1 - lse_desc,
                                                    -2 - lse_desc], rtol=0, atol=1e-12)
        assert vals[0, p, 4] == -np.inf
    # row 0 at T = 0.5: scaled [2, 6, 6, -inf, 0, 4]; the argmax is the lower 6
    lse = math.log(2 + math.exp(-4) + math.exp(-6) + math.exp(-2))
    assert list(ids[1, 0]) == [1, 1, 2, 5, 0]
    np.testing.assert_allclose(vals[1, 0, :4], [-lse, -lse, -lse, -2 - lse], rtol=0, atol=1e-12)
    assert list(ranks.ravel()) == [1, 1, 1, -1]
    assert np.all(ids[1, 1] == -1) and np.all(np.isnan(vals[1, 1]))   # p >= valid[1]


def _batch(seed, vocab=777, m=5, canvas=4):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((m * canvas, vocab)) * 2).astype(np.float32)
    x[rng.random(x.shape) < 0.2] = -np.inf
    x[3] = np.round(x[3])                         # ties
    x[5] = 0.5                                    # constant
    x[6] = -np.inf                                # all -inf
    src = rng.permutation(m).astype(np.int32)
    slots = rng.permutation(m + 2)[:m].astype(np.int32)
    keep = np.array([1, 0, 1, 1, 1], np.uint8)[:m]
    valid = np.array([4, 4, 2, 0, 3], np.int32)[:m]
    temps = np.array([1.0, 0.7, 0.0, 1e-3, 1.3], np.float32)[:m]
    return x, src, slots, keep, valid, temps, m, canvas


@pytest.mark.parametrize("seed", [0, 1])
def test_topk_columns_match_the_topk_routine(seed):
    x, src, slots, keep, valid, temps, m, canvas = _batch(seed)
    k, width = 6, 9
    ids, vals, ranks = oracle.stash(x, canvas, src, slots, keep, valid, temps, k, None, None,
                                    m + 2, width)
    for j in range(m):
        for p in range(canvas):
            out = ids[slots[j], p]
            if not keep[j] or p >= valid[j]:
                assert np.all(out == -1) and ranks[slots[j], p] == -1
                continue
            row = src[j] * canvas + p
            ri, rl = oracle.topk_rows(np.ascontiguousarray(x[row:row + 1]), temps[j:j + 1], k)
            assert out[0] == ri[0, 0] and list(out[1:1 + k]) == list(ri[0])
            np.testing.assert_allclose(vals[slots[j], p, 1:1 + k], rl[0], rtol=0, atol=1e-9)
            assert list(out[1 + k:]) == [0] * (width - 1 - k)
            assert np.all(vals[slots[j], p, 1 + k:] == -np.inf)
            # out_ranks: the pages do not say what the rank counts, so it has no
            # pin here (parity unpinned); only that a written row has one
            assert ranks[slots[j], p] != -1


def test_token_ids_values_and_logits_mode():
    """The token-id path against a numpy log-softmax; a request without ids
    (count 0) takes the top-k; ids outside the vocabulary give NaN; logits
    mode writes x / T in fp32 exactly."""
    x, src, slots, keep, valid, temps, m, canvas = _batch(7, vocab=300)
    tok = np.array([[5, 299, 0, 17], [1, 2, 3, 4], [9, 9, 300, -1], [0, 0, 0, 0], [42, 7, 7, 1]],
                   np.int32)
    nti = np.array([4, 2, 4, 1, 0], np.int32)
    width, k = 7, 3
    for mode in (False, True):
        ids, vals, _ = oracle.stash(x, canvas, src, slots, keep, valid, temps, k, nti, tok, m + 2,
                                    width, logits_mode=mode)
        for j in range(m):
            for p in range(min(valid[j], canvas)):
                if not keep[j]:
                    continue
                row = src[j] * canvas + p
                s, lp = _log_softmax(x[row], temps[j])
                out, v = ids[slots[j], p], vals[slots[j], p]
                if nti[j] > 0:
                    listed = list(tok[j, :nti[j]])[:width - 1]
                else:
                    listed = list(oracle.topk_rows(np.ascontiguousarray(x[row:row + 1]),
                                                   temps[j:j + 1], k)[0][0])
                assert list(out[1:1 + len(listed)]) == listed
                for c, t in enumerate(listed, start=1):
                    if not 0 <= t < x.shape[1]:
                        assert np.isnan(v[c])
                    elif mode:
                        assert v[c] == float(s[t])
                    elif np.isfinite(np.max(s)):
                        assert (lp[t] == -np.inf and v[c] == -np.inf) or abs(v[c] - lp[t]) <= 1e-9
                    else:
                        assert np.isnan(v[c])
                assert np.all(out[1 + len(listed):] == 0)


def test_token_count_past_the_list_is_the_list():
    """A request's token-id list has ids_stride entries: a count above that
    gives the same stash as a count equal to it (the rest is padding)."""
    x, src, slots, keep, valid, temps, m, canvas = _batch(5, vocab=300)
    tok = np.array([[5, 299, 0, 17], [1, 2, 3, 4], [9, 9, 30, 1], [0, 0, 0, 0], [42, 7, 7, 1]],
                   np.int32)
    over = np.array([4, 9, 4, 1, 7], np.int32)
    exact = np.minimum(over, tok.shape[1]).astype(np.int32)
    a = oracle.stash(x, canvas, src, slots, keep, valid, temps, 3, over, tok, m + 2, 9)
    b = oracle.stash(x, canvas, src, slots, keep, valid, temps, 3, exact, tok, m + 2, 9)
    for u, v in zip(a, b):
        assert np.array_equal(u, v, equal_nan=True) if u.dtype.kind == "f" else np.array_equal(u, v)
    j = int(np.flatnonzero((keep != 0) & (valid > 0) & (over > tok.shape[1]))[0])
    out = a[0][slots[j], 0]
    assert list(out[1:5]) == list(tok[j]) and np.all(out[5:] == 0)


def test_width_truncates_and_no_topk():
    x, src, slots, keep, valid, temps, m, canvas = _batch(3)
    ids, vals, _ = oracle.stash(x, canvas, src, slots, keep, valid, temps, 10, None, None, m + 2, 3)
    ids0, _, _ = oracle.stash(x, canvas, src, slots, keep, valid, temps, 0, None, None, m + 2, 3)
    j = 0
    assert keep[j] and valid[j] > 0
    row = src[j] * canvas
    ri, _ = oracle.topk_rows(np.ascontiguousarray(x[row:row + 1]), temps[:1], 2)
    assert list(ids[slots[j], 0]) == [ri[0, 0], ri[0, 0], ri[0, 1]]
    assert list(ids0[slots[j], 0]) == [ri[0, 0], 0, 0]
