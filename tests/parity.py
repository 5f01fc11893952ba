"""Comparison rules between the CUDA library and the CPU oracle.

Tolerances (fixed by the acceptance criteria of the method):
  - argmax, top-k ids: bit-exact;
  - sample: exact, except rows whose two best noisy scores (oracle, double)
    are within NEAR_TIE_REL * max(1, |best|) -- the GPU scores in fp32 --
    which are counted, not failed;
  - entropy: ENTROPY_ABS absolute;
  - logprobs: LOGPROB_ABS absolute, or one fp32 ulp of the oracle value
    rounded to fp32 when that is larger (|lp| up to 1e10 at T = 1e-10);
  - probs: one unit in the last place of bf16 / fp16 (codes of non-negative
    numbers are ordered like the numbers, so one ulp is a code distance of
    one); NaN where the oracle has NaN.
"""
from __future__ import annotations

import numpy as np

NEAR_TIE_REL = 1e-5
ENTROPY_ABS = 1e-4
LOGPROB_ABS = 1e-4
GUMBEL_ABS = 1e-5


def _nan_code(c, dtype_code):
    c = c.astype(np.int64)
    if dtype_code == 1:   # bf16
        return ((c & 0x7F80) == 0x7F80) & ((c & 0x007F) != 0)
    return ((c & 0x7C00) == 0x7C00) & ((c & 0x03FF) != 0)


def check_row_stats(gpu: dict, ref: dict, probs_dtype: int, where: str = ""):
    """gpu: numpy dict (argmax, sample, entropy, probs codes or None) for the
    same rows as ref (an oracle dict). Returns the number of near-tie sample
    mismatches; raises AssertionError on any other difference."""
    a_g, a_r = gpu["argmax"], ref["argmax"]
    bad = np.flatnonzero(a_g != a_r)
    assert bad.size == 0, f"{where} argmax differs at rows {bad[:10]}: {a_g[bad[:10]]} vs {a_r[bad[:10]]}"

    s_g, s_r = gpu["sample"], ref["sample"]
    diff = np.flatnonzero(s_g != s_r)
    near = ref["sample_gap"][diff] <= NEAR_TIE_REL * np.maximum(1.0, np.abs(ref["sample_best"][diff]))
    hard = diff[~near]
    assert hard.size == 0, (f"{where} sample differs at non-tie rows {hard[:10]}: "
                            f"{s_g[hard[:10]]} vs {s_r[hard[:10]]}, gaps {ref['sample_gap'][hard[:10]]}")

    e_g, e_r = gpu["entropy"].astype(np.float64), ref["entropy"]
    err = np.abs(e_g - e_r)
    worst = int(np.argmax(err)) if err.size else 0
    assert err.size == 0 or err[worst] <= ENTROPY_ABS, (
        f"{where} entropy error {err[worst]:.3e} at row {worst}: {e_g[worst]} vs {e_r[worst]}")

    if probs_dtype:
        p_g, p_r = gpu["probs"].astype(np.int64), ref["probs"].astype(np.int64)
        nan_r = _nan_code(ref["probs"], probs_dtype)
        nan_g = _nan_code(gpu["probs"], probs_dtype)
        assert np.array_equal(nan_r, nan_g), f"{where} NaN probabilities differ"
        d = np.abs(p_g - p_r)
        d[nan_r] = 0
        if d.size and d.max() > 1:
            r, c = np.unravel_index(int(np.argmax(d)), d.shape)
            raise AssertionError(f"{where} probs differ by {d.max()} codes at row {r} col {c}: "
                                 f"{p_g[r, c]:#06x} vs {p_r[r, c]:#06x}")
    return int(near.sum())


def check_topk(ids_g, lp_g, ids_r, lp_r, where: str = ""):
    """Top-k rows: ids exact; logprobs within LOGPROB_ABS or one fp32 ulp."""
    bad = np.flatnonzero(np.any(ids_g != ids_r, axis=1))
    assert bad.size == 0, f"{where} top-k ids differ at rows {bad[:5]}: {ids_g[bad[0]]} vs {ids_r[bad[0]]}"
    ref32 = lp_r.astype(np.float32)
    both_nan = np.isnan(lp_g) & np.isnan(lp_r)
    both_ninf = np.isneginf(lp_g) & np.isneginf(lp_r)
    tol = np.maximum(LOGPROB_ABS, np.spacing(np.abs(ref32)).astype(np.float64))
    with np.errstate(invalid="ignore"):
        ok = both_nan | both_ninf | (np.abs(lp_g.astype(np.float64) - lp_r) <= tol)
    if not ok.all():
        r, c = np.argwhere(~ok)[0]
        raise AssertionError(f"{where} logprob row {r} rank {c}: {lp_g[r, c]!r} vs {lp_r[r, c]!r}")
