"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a library routine, a closed form, an
invariant of the method, or a statistical law, so that a plausible slip in
the oracle (a dropped term, a wrong sign or index, a swapped operand) fails
at least one of them. CPU only.
"""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import PROBS_BF16, PROBS_FP16, PROBS_NONE

LN2_NEG_LOG = 0.36651292058166435  # -ln(ln 2): Gumbel noise at u = 1/2


# ----------------------------------------------------------------- Philox

def _curand():
    cands = [ctypes.util.find_library("curand"),
             "/usr/local/cuda/lib64/libcurand.so",
             "/usr/local/cuda/targets/sbsa-linux/lib/libcurand.so",
             "/usr/local/cuda/targets/x86_64-linux/lib/libcurand.so"]
    for c in cands:
        if c and (os.path.exists(c) or not c.startswith("/")):
            try:
                return ctypes.CDLL(c)
            except OSError:
                continue
    return None


def _curand_host_philox_words(lib, seed, n):
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) != 0:
        pytest.skip("curandCreateGeneratorHost failed")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        buf = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, ctypes.c_void_p(buf.ctypes.data), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return buf


@pytest.mark.parametrize("seed", [0, 0x123456789ABCDEF0, 2**64 - 1, 42])
def test_philox_matches_curand_host_generator(seed):
    """cuRAND's host PHILOX4_32_10 generator is an independent Philox4x32-10.

    Its host ordering emits, for output word w with block b = w // 4, word
    w % 4 of the block at counter (b // 65536, 0, b % 65536, 0) under key
    (lo32(seed), hi32(seed)). In the oracle's layout that block is column
    group b // 65536 of row b % 65536, so the first 3 * 65536 blocks cover
    columns 0..11 of rows 0..65535: every counter word but the last gets
    exercised, and the key schedule by three seeds.
    """
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    groups = 3
    words = _curand_host_philox_words(lib, seed, 65536 * 4 * groups)
    # [group, row, word] -> [row, group * 4 + word]
    ref = words.reshape(groups, 65536, 4).transpose(1, 0, 2).reshape(65536, groups * 4)
    bits, _ = oracle.philox_gumbel(seed, 0, 65536, groups * 4)
    assert np.array_equal(bits, ref)


def test_philox_block_layout():
    """noise_bits(seed, row, col) is word col % 4 of the block at counter
    (col // 4, 0, row, 0): one Philox call serves four neighbouring columns,
    and high row bits land in the fourth counter word."""
    seed = 0x0123456789ABCDEF
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for row, col in [(0, 0), (5, 7), (65535, 1023), (2**32 + 3, 6), (7, 2**33 + 1)]:
        grp = col // 4
        block = oracle.philox4x32_10([grp & 0xFFFFFFFF, grp >> 32, row & 0xFFFFFFFF, row >> 32], key)
        assert oracle.noise_bits(seed, row, col) == block[col % 4]


def test_philox_bits_balanced_and_uniform():
    from scipy import stats
    bits, _ = oracle.philox_gumbel(1234, 0, 512, 512)
    flat = bits.ravel()
    n = flat.size
    for b in range(32):
        ones = int(((flat >> np.uint32(b)) & 1).sum())
        assert abs(ones - n / 2) < 5 * math.sqrt(n / 4), b
    top = (flat >> np.uint32(24)).astype(np.int64)
    counts = np.bincount(top, minlength=256)
    assert stats.chisquare(counts).pvalue > 1e-4


# ---------------------------------------------------------- noise mapping

def test_uniform_mapping_endpoints():
    assert oracle.uniform(0x00000000) == np.float32(1e-20)   # clamp(min=1e-20)
    assert oracle.uniform(0x000000FF) == np.float32(1e-20)   # low 8 bits unused
    assert oracle.uniform(0x00000100) == 2.0 ** -24
    assert oracle.uniform(0x80000000) == 0.5
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24


def test_gumbel_point_values():
    assert abs(oracle.gumbel_of_bits(0x80000000) - LN2_NEG_LOG) < 1e-15
    # u = 1e-20f: -log(-log u) with -log u = 46.05..., so g ~ -3.83
    u = float(np.float32(1e-20))
    assert abs(oracle.gumbel_of_bits(0) - (-math.log(-math.log(u)))) < 1e-12
    assert oracle.gumbel_of_bits(0) < -3.82
    # u = 1 - 2^-24: the largest noise, ~16.636
    assert 16.63 < oracle.gumbel_of_bits(0xFFFFFFFF) < 16.64


def test_gumbel_distribution_ks():
    """The noise follows the standard Gumbel law (scipy's gumbel_r)."""
    from scipy import stats
    _, g = oracle.philox_gumbel(99, 0, 256, 1024)
    res = stats.kstest(g.ravel(), stats.gumbel_r.cdf)
    assert res.pvalue > 1e-3


# ------------------------------------------------------ dtype conversions

def _conversion_probe_values():
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000).astype(np.float32),
            (rng.random(20000) * 1e-3).astype(np.float32),
            np.float32(2.0) ** rng.integers(-149, 127, 20000).astype(np.float32),
            rng.random(20000).astype(np.float32) * np.float32(2.0 ** -130)]
    v = np.concatenate(vals)
    # exact halfway cases for bf16 (low 16 bits 0x8000) and fp16
    halves = (rng.integers(0, 2**16, 5000, dtype=np.uint32) << 16 | 0x8000).astype(np.uint32)
    v = np.concatenate([v, halves.view(np.float32),
                        np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 65504.0, 65520.0, 6e-8, 3e-8,
                                  2.0 ** -24, 2.0 ** -25, 3.4e38], dtype=np.float32)])
    return v[np.isfinite(v) | np.isinf(v)]


def test_bf16_rounding_matches_torch():
    v = _conversion_probe_values()
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16_bits(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_fp16_rounding_matches_numpy():
    v = _conversion_probe_values()
    with np.errstate(over="ignore"):  # the probe values include overflow to inf on purpose
        ref = v.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16_bits(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- helpers

def _rows(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def _bf16_to_f32(codes):
    return (codes.astype(np.uint32) << 16).view(np.float32)


def _tiny_inputs(rows=64, vocab=8192, seed=0):
    import workloads
    w = workloads.make("tiny", rows=rows)
    return w["logits"].numpy(), w["temps"].numpy(), w["canvas_len"]


# -------------------------------------------------------------- row stats

def test_argmax_matches_numpy_on_ties():
    x, temps, W = _tiny_inputs()
    r = oracle.row_stats(x, temps, W, seed=0, probs_dtype=PROBS_NONE, threads=4)
    te = np.maximum(np.repeat(temps, W), np.float32(1e-10)).astype(np.float32)
    scaled = (x / te[:, None]).astype(np.float32)   # IEEE fp32 division
    assert np.array_equal(r["argmax"], np.argmax(scaled, axis=1))


def test_greedy_rows_sample_the_argmax():
    x, temps, W = _tiny_inputs()
    temps = temps.copy()
    temps[1] = -0.5          # T <= 0 is greedy as well
    r = oracle.row_stats(x, temps, W, seed=3, probs_dtype=PROBS_NONE, threads=4)
    greedy = np.repeat(temps <= 0, W)
    assert greedy.sum() == 2 * W
    assert np.array_equal(r["sample"][greedy], r["argmax"][greedy])
    assert np.all(np.isinf(r["sample_gap"][greedy]))
    # with noise, the sample differs from the argmax on some rows
    assert np.any(r["sample"][~greedy] != r["argmax"][~greedy])


@pytest.mark.parametrize("vocab", [8192, 131072, 262144])
def test_constant_row_entropy_is_log_v(vocab):
    x = np.full((1, vocab), 0.37, dtype=np.float32)
    for t in (0.0, 0.7, 1.0):
        r = oracle.row_stats(x, np.array([t], np.float32), 1, seed=5, probs_dtype=PROBS_BF16)
        assert abs(r["entropy"][0] - math.log(vocab)) < 1e-12
        assert r["argmax"][0] == 0
        p = _bf16_to_f32(r["probs"][0])
        assert np.all(p == np.float32(1.0 / vocab))     # a power of two: exact


@pytest.mark.parametrize("t", [0.0, 1e-10, 1e-3, 1.0, 1.3])
def test_one_hot_row(t):
    vocab, hot = 4099, 1234
    x = np.full((1, vocab), -np.inf, dtype=np.float32)
    x[0, hot] = 0.0
    r = oracle.row_stats(x, np.array([t], np.float32), 1, seed=11, probs_dtype=PROBS_FP16)
    assert r["argmax"][0] == hot and r["sample"][0] == hot
    assert r["entropy"][0] == 0.0
    p = r["probs"][0]
    assert p[hot] == 0x3C00 and np.count_nonzero(p) == 1    # fp16 1.0 and zeros


@pytest.mark.parametrize("k,a,b", [(1, 3.0, 0.0), (7, 0.0, -2.5), (100, 1.25, 1.0)])
def test_two_level_entropy_closed_form(k, a, b):
    vocab = 1000
    x = np.full((1, vocab), b, dtype=np.float32)
    x[0, 500:500 + k] = a
    r = oracle.row_stats(x, np.array([1.0], np.float32), 1, seed=0, probs_dtype=PROBS_NONE)
    p1 = 1.0 / (k + (vocab - k) * math.exp(b - a))
    p2 = p1 * math.exp(b - a)
    h = -k * p1 * math.log(p1) - (vocab - k) * p2 * math.log(p2)
    assert abs(r["entropy"][0] - h) < 1e-12
    assert r["argmax"][0] == (500 if a > b else 0)


def test_entropy_two_formulas_agree():
    x, temps, W = _tiny_inputs()
    r = oracle.row_stats(x, temps, W, seed=0, probs_dtype=PROBS_NONE, threads=4)
    assert np.max(np.abs(r["entropy"] - r["entropy_check"])) < 1e-9


def test_entropy_matches_torch_float64_log_softmax():
    """Library pin: torch.log_softmax in float64 on the fp32-scaled row."""
    x, temps, W = _tiny_inputs()
    r = oracle.row_stats(x, temps, W, seed=0, probs_dtype=PROBS_NONE, threads=4)
    te = np.maximum(np.repeat(temps, W), np.float32(1e-10)).astype(np.float32)
    scaled = torch.from_numpy((x / te[:, None]).astype(np.float32)).double()
    lp = torch.log_softmax(scaled, dim=-1)
    p = lp.exp()
    h = -torch.where(p > 0, p * lp, torch.zeros_like(p)).sum(-1).numpy()
    assert np.max(np.abs(r["entropy"] - h)) < 1e-9


def test_masked_columns_drop_out():
    rng = np.random.default_rng(1)
    v = 3000
    x = (rng.standard_normal(v) * 3).astype(np.float32)
    mask = rng.random(v) < 0.3
    xm = x.copy()
    xm[mask] = -np.inf
    r_full = oracle.row_stats(xm[None], np.array([0.8], np.float32), 1, 0, PROBS_BF16)
    r_cmp = oracle.row_stats(_rows(x[~mask][None]), np.array([0.8], np.float32), 1, 0, PROBS_BF16)
    assert abs(r_full["entropy"][0] - r_cmp["entropy"][0]) < 1e-12
    assert np.array_equal(r_full["probs"][0][~mask], r_cmp["probs"][0])
    assert np.all(r_full["probs"][0][mask] == 0)
    assert np.flatnonzero(~mask)[r_cmp["argmax"][0]] == r_full["argmax"][0]


def test_power_of_two_temperature_is_exact_rescaling():
    x, _, _ = _tiny_inputs(rows=8)
    t1 = oracle.row_stats(x, np.array([1.0], np.float32), 8, 9, PROBS_BF16)
    t2 = oracle.row_stats(_rows(x * 2), np.array([2.0], np.float32), 8, 9, PROBS_BF16)
    for key in ("argmax", "sample", "entropy"):
        assert np.array_equal(t1[key], t2[key]), key
    assert np.array_equal(t1["probs"], t2["probs"])


def test_probs_sum_to_one():
    x, temps, W = _tiny_inputs()
    r = oracle.row_stats(x, temps, W, seed=0, probs_dtype=PROBS_BF16, threads=4)
    s = _bf16_to_f32(r["probs"]).astype(np.float64).sum(axis=1)
    # each bf16 code is within 2^-9 (relative) of its probability
    assert np.all(np.abs(s - 1.0) <= 2.0 ** -9)


def test_all_neg_inf_row():
    x = np.full((2, 64), -np.inf, dtype=np.float32)
    r = oracle.row_stats(x, np.array([1.0], np.float32), 2, 0, PROBS_BF16)
    assert list(r["argmax"]) == [0, 0] and list(r["sample"]) == [0, 0]
    assert list(r["entropy"]) == [0.0, 0.0]
    assert np.all(np.isnan(_bf16_to_f32(r["probs"])))


def test_row_subsets_are_independent():
    x, temps, W = _tiny_inputs(rows=32)
    full = oracle.row_stats(x, temps, W, seed=17, probs_dtype=PROBS_BF16)
    part = oracle.row_stats(x, temps, W, seed=17, probs_dtype=PROBS_BF16, rows_sel=[3, 20, 31])
    for key in ("argmax", "sample", "entropy"):
        assert np.array_equal(full[key][[3, 20, 31]], part[key][[3, 20, 31]])


@pytest.mark.parametrize("t", [1.0, 0.5])
def test_gumbel_max_frequencies_follow_softmax(t):
    """Gumbel-max on V = 8: 10^5 rows (independent noise) sample
    softmax(x / T); chi-square at p > 0.001."""
    from scipy import stats
    x = np.array([0.3, -1.0, 2.0, 0.0, 1.1, -0.4, 0.7, 1.5], dtype=np.float32)
    n = 100_000
    logits = np.tile(x, (n, 1))
    r = oracle.row_stats(logits, np.array([t], np.float32), n, seed=2024, threads=8)
    counts = np.bincount(r["sample"], minlength=8)
    s = x.astype(np.float64) / np.float32(t)
    p = np.exp(s - s.max())
    p /= p.sum()
    assert stats.chisquare(counts, p * n).pvalue > 1e-3


def test_gumbel_max_constant_row_is_uniform():
    from scipy import stats
    n, v = 64_000, 16
    logits = np.full((n, v), 1.5, dtype=np.float32)
    r = oracle.row_stats(logits, np.array([0.9], np.float32), n, seed=7, threads=8)
    counts = np.bincount(r["sample"], minlength=v)
    assert stats.chisquare(counts).pvalue > 1e-3
    assert np.all(r["argmax"] == 0)


def test_sample_gap_and_best_match_a_numpy_ranking():
    """The near-tie classifier the parity tests rely on: for every noisy row
    the oracle's sample, best score and gap (best minus second-best) equal a
    numpy ranking of the scores x / T (fp32 quotient) + g, with g computed
    here from the Philox words (u = max((w >> 8) 2^-24, 1e-20f), g =
    -log(-log u)); greedy rows report an infinite gap and the max."""
    x, temps, W = _tiny_inputs()
    rows, vocab = x.shape
    seed = 31
    r = oracle.row_stats(x, temps, W, seed=seed, threads=8)
    bits, _ = oracle.philox_gumbel(seed, 0, rows, vocab)
    u = np.maximum((bits >> 8).astype(np.float32) * np.float32(2.0 ** -24), np.float32(1e-20))
    g = -np.log(-np.log(u.astype(np.float64)))
    for i in range(rows):
        t = temps[i // W]
        s = (x[i] / np.float32(max(t, 1e-10))).astype(np.float32).astype(np.float64)
        if t <= 0:
            assert r["sample_gap"][i] == np.inf and r["sample_best"][i] == s.max()
            continue
        score = s + g[i]
        order = np.argsort(-score, kind="stable")
        best, second = score[order[0]], score[order[1]]
        assert r["sample"][i] == order[0]
        assert abs(r["sample_best"][i] - best) <= 1e-12 * max(1.0, abs(best))
        assert abs(r["sample_gap"][i] - (best - second)) <= 1e-12 * max(1.0, abs(best))


# ------------------------------------------------------------------ top-k

def _stable_topk(x, te, k):
    s = (x / te).astype(np.float32) + np.float32(0.0)
    order = np.argsort(-s, kind="stable")[:k]
    return order, s


def test_topk_matches_stable_argsort_and_scipy_logsumexp():
    from scipy.special import logsumexp
    x, temps, W = _tiny_inputs()
    keep = np.ones(temps.size, np.uint8)
    k = 8
    ids, lps = oracle.topk_logprobs(x, temps, W, keep, k, threads=4)
    for i in range(x.shape[0]):
        te = np.float32(max(np.float32(temps[i // W]), np.float32(1e-10)))
        order, s = _stable_topk(x[i], te, k)
        assert np.array_equal(ids[i], order), i
        ref = s[order].astype(np.float64) - logsumexp(s.astype(np.float64))
        assert np.max(np.abs(lps[i] - ref)) < 1e-6 * max(1.0, np.max(np.abs(ref))), i


def test_topk_constant_row():
    v = 4096
    x = np.full((1, v), -2.0, dtype=np.float32)
    ids, lps = oracle.topk_logprobs(x, np.array([0.7], np.float32), 1, np.ones(1, np.uint8), 20)
    assert list(ids[0]) == list(range(20))
    assert np.allclose(lps[0], -math.log(v), atol=1e-12, rtol=0)


def test_topk_one_hot_row():
    v, hot = 1000, 321
    x = np.full((1, v), -np.inf, dtype=np.float32)
    x[0, hot] = 0.0
    ids, lps = oracle.topk_logprobs(x, np.array([0.0], np.float32), 1, np.ones(1, np.uint8), 5)
    assert list(ids[0]) == [hot, 0, 1, 2, 3]
    assert lps[0, 0] == 0.0 and np.all(np.isneginf(lps[0, 1:]))


def test_topk_signed_zero_is_one_value():
    x = np.full((1, 16), -1.0, dtype=np.float32)
    x[0, 9] = 0.0
    x[0, 2] = -0.0
    ids, _ = oracle.topk_logprobs(x, np.array([1.0], np.float32), 1, np.ones(1, np.uint8), 3)
    assert list(ids[0]) == [2, 9, 0]


def test_topk_skips_rows_of_slots_not_kept():
    x, temps, W = _tiny_inputs()
    keep = np.array([1, 0, 1, 0], np.uint8)
    ids, lps = oracle.topk_logprobs(x, temps, W, keep, 8, threads=4)
    kept_rows = np.repeat(keep.astype(bool), W)
    assert np.all(ids[~kept_rows] == -1) and np.all(np.isnan(lps[~kept_rows]))
    assert np.all(ids[kept_rows] >= 0)


def test_topk_zero_temperature_clamps():
    """T = 0 divides by 1e-10f (the row-stats clamp): logprobs stay finite
    for the top element and the order is the order of the logits."""
    x = np.array([[0.5, 0.25, 0.5 + 2**-20, -1.0]], dtype=np.float32)
    ids, lps = oracle.topk_logprobs(x, np.array([0.0], np.float32), 1, np.ones(1, np.uint8), 4)
    assert list(ids[0]) == [2, 0, 1, 3]
    assert lps[0, 0] == 0.0
    assert lps[0, 1] < -1e3
