"""GPU parity of drs_row_stats against the CPU oracle (same bytes in).

Small cases compare every row; the full-size workloads compare sampled rows
(the oracle computes them one by one) in the launch configuration the
benchmark times.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import drs, gpu_row_stats, oracle_rows, sample_rows, subset
from parity import check_row_stats

pytestmark = pytest.mark.gpu

BF16, FP16, NONE = 1, 2, 0


def _dev(x):
    return torch.as_tensor(x).cuda()


def _compare(logits_dev, temps, canvas_len, seed, probs_dtype, rows_sel=None, row0=0, where=""):
    rows = logits_dev.shape[0]
    g = gpu_row_stats(logits_dev, _dev(temps), canvas_len, seed, probs_dtype, row0=row0)
    rows_sel = np.arange(rows) if rows_sel is None else np.asarray(rows_sel)
    r = oracle_rows(logits_dev, temps, canvas_len, seed, probs_dtype, rows_sel, row0=row0)
    return check_row_stats(subset(g, rows_sel), r, probs_dtype, where)


@pytest.mark.parametrize("seed", [0, 12345, 2**63 + 7])
def test_tiny_workload_every_row(seed):
    w = workloads.make("tiny")
    near = _compare(w["logits"].cuda(), w["temps"].numpy(), w["canvas_len"], seed, BF16,
                    where=f"tiny seed {seed}")
    assert near <= 2


@pytest.mark.parametrize("vocab", [1, 2, 3, 4, 5, 7, 17, 1000, 4097, 8191, 16384, 16385,
                                   40003, 70001, 131072])
@pytest.mark.parametrize("pad", [0, 1, 4])
def test_shapes_and_strides(vocab, pad):
    """Ragged vocabularies (tails of 1-3 columns, chunks shared by several
    CTAs) and row strides that are not multiples of 4 (no bulk copy)."""
    rows, canvas = 12, 4
    rng = np.random.default_rng(vocab * 7 + pad)
    buf = (rng.standard_normal((rows, vocab + pad)) * 2.5).astype(np.float32)
    buf[:, vocab:] = np.nan                         # never read
    buf[:, :vocab][rng.random((rows, vocab)) < 0.1] = -np.inf
    buf[0, :vocab] = -np.inf                        # a row that is -inf everywhere
    if vocab > 1:
        buf[1, :vocab] = 0.75                       # constant row
    temps = np.array([0.0, 0.7, 1.0, 1e-3], np.float32)
    dev = _dev(buf)[:, :vocab]
    for probs in (BF16, FP16, NONE):
        _compare(dev, temps, canvas, 99, probs, where=f"V={vocab} pad={pad} probs={probs}")


def test_special_rows_on_a_shared_row():
    """One-hot, constant, all -inf and ordinary rows at V = 131072 (16
    tiles of a row merged) under every temperature regime."""
    vocab = 131072
    rng = np.random.default_rng(5)
    rows = 16
    x = (rng.standard_normal((rows, vocab)) * 3).astype(np.float32)
    x[0] = -np.inf
    x[0, 77777] = 0.0                 # one-hot in a middle chunk
    x[1] = 1.25                       # constant
    x[2] = -np.inf                    # all -inf
    x[3, 5] = x[3, 100000] = 50.0     # tied maxima in different chunks
    x[4, :] = -np.inf
    x[4, 131071] = -3.0               # one-hot at the last column
    temps = np.array([0.0, 1e-10, 1e-3, 1.0], np.float32)
    for canvas in (4, 1):
        t = temps if canvas == 4 else np.resize(temps, rows)
        _compare(_dev(x), t, canvas, 7, BF16, where=f"special canvas={canvas}")


def test_zero_rows_is_a_no_op():
    import vocab_row_sampling_gb300 as drs
    x = torch.empty(0, 100, device="cuda")
    a, s, e, p = drs.row_stats(x, torch.ones(1, device="cuda"), 1, 0, torch.bfloat16)
    assert a.numel() == 0 and p.shape == (0, 100)


def test_row0_offsets_equal_one_call():
    """A batch split in two calls with row0 gives the one-call result."""
    w = workloads.make("tiny")
    x = w["logits"].cuda()
    t = w["temps"].cuda()
    whole = gpu_row_stats(x, t, 16, 3, BF16)
    a = gpu_row_stats(x[:32], t, 16, 3, BF16, row0=0)
    b = gpu_row_stats(x[32:], t, 16, 3, BF16, row0=32)
    for k in ("argmax", "sample", "entropy", "probs"):
        assert np.array_equal(np.concatenate([a[k], b[k]]), whole[k]), k


def test_repeated_calls_are_deterministic():
    w = workloads.make("tiny")
    x = w["logits"].cuda()
    t = w["temps"].cuda()
    one = gpu_row_stats(x, t, 16, 11, BF16)
    for _ in range(3):
        again = gpu_row_stats(x, t, 16, 11, BF16)
        for k in ("argmax", "sample", "entropy", "probs"):
            assert np.array_equal(one[k], again[k]), k


@pytest.mark.parametrize("which", ["400000", "368640", "368641", "491520", "1000003", "max"])
def test_long_rows(which):
    """Rows of many tiles with a ragged last one: 400000 columns; 368640, the
    longest rows of the merge's short-row instantiation (60 pass-1 tiles),
    and one column more; 491520 (60 pass-2 tiles); 1000003 columns; the
    largest supported vocabulary."""
    import vocab_row_sampling_gb300 as drs
    vocab = drs.DRS_MAX_VOCAB if which == "max" else int(which)
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((3, vocab)) * 3).astype(np.float32)
    x[2, vocab - 1] = 40.0
    _compare(_dev(x), np.array([0.9, 0.0, 1.1], np.float32), 1, 5, BF16, where=which)


def test_raw_and_exact_domains_in_one_row():
    """Scaled logits around the magnitude 256 at which a warp switches from
    working on the raw logits to dividing every logit exactly: the warps of
    one row then mix both, with probabilities far from negligible."""
    rng = np.random.default_rng(5)
    rows, vocab = 8, 70001
    x = (250.0 + rng.random((rows, vocab)) * 12.0).astype(np.float32)
    x[1] = -x[1]                                   # negative side of the switch
    x[2, ::7] = 256.0                              # ties at the switch itself
    x[3] = (rng.standard_normal(vocab) * 3).astype(np.float32)
    x[3, 40000:] += 255.0                          # half raw, half exact
    temps = np.array([1.0, 1.0, 0.999, 1.001, 1.0, 0.5, 1.0, 2.0], np.float32)
    for seed in (3, 4):
        _compare(_dev(x), temps, 1, seed, BF16, where=f"domains seed {seed}")


# ------------------------------------------------------------- full sizes

def _full(name, n_sample, seeds=None, always=()):
    w = workloads.make(name, device="cuda")
    V = w["vocab"]
    view = w["logits"][:, :V]
    rows = w["rows"]
    sel = sample_rows(rows, n_sample, seed=1, always=always)
    near = 0
    for seed in (seeds or w["seeds"]):
        near += _compare(view, w["temps"].cpu().numpy(), w["canvas_len"], seed, w["probs_dtype"],
                         rows_sel=sel, where=f"{name} seed {seed}")
    del w, view
    torch.cuda.empty_cache()
    return near


@pytest.mark.slow
def test_adversarial_workload_sampled_rows():
    w = workloads.make("adversarial", device="cuda")
    x = w["logits"]
    finite = torch.isfinite(x).sum(1)
    const = (x.max(1).values == x.min(1).values).nonzero().flatten()[:12].tolist()
    onehot = (finite == 1).nonzero().flatten()[:12].tolist()
    del w, x, finite
    torch.cuda.empty_cache()
    _full("adversarial", 96, always=const + onehot)


@pytest.mark.slow
def test_step_workload_sampled_rows():
    _full("step", 24, always=[0, 255, 256, 2047])


@pytest.mark.slow
def test_strided_workload_sampled_rows_all_seeds():
    _full("strided", 6, always=[0, 2047])


@pytest.mark.slow
def test_large_workload_sampled_rows():
    w = workloads.make_temps_keep("large")[0]
    zero_slots = np.flatnonzero(w.numpy() == 0)
    always = [int(s) * 256 + 3 for s in zero_slots[:3]]
    _full("large", 12, always=always)


def test_kernel_timing_hook_counts_calls():
    """The measurement hook: with timing on, each call records its five row
    kernels; the averages are positive and the count is the number of calls;
    with timing off, calls are not recorded."""
    lib = drs()
    w = workloads.make("tiny")
    x, t = w["logits"].cuda(), w["temps"].cuda()
    lib.drs_kernel_timing(True)
    for _ in range(3):
        lib.row_stats(x, t, 16, 0, torch.bfloat16)
    lib.drs_kernel_timing(False)
    lib.row_stats(x, t, 16, 0, torch.bfloat16)
    times, calls = lib.drs_kernel_times()
    assert calls == 3
    assert set(times) == set(lib.KERNEL_NAMES)
    assert all(v > 0.0 for v in times.values()), times
