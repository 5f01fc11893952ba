"""CPU oracle for the DiffusionGemma per-row sampler statistics.

TEST INFRASTRUCTURE. This package is a plain, slow, obviously correct
restatement of what the sampler computes (see ``drs_oracle.c`` for the
passages it follows and the readings taken where the pages are silent). Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import it. The CUDA library never calls it and shares no
code with it.

Parallelism: each C call handles a row range single-threaded; ``threads > 1``
splits the rows over a thread pool (ctypes releases the GIL), which changes
nothing in the arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "drs_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

PROBS_NONE, PROBS_BF16, PROBS_FP16 = 0, 1, 2

# Flags: IEEE fp32 division and double arithmetic exactly as written -- no
# contraction into FMA (GCC contracts by default on aarch64), no fast-math.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    c_i64, c_u64, c_i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32
    vp = ctypes.c_void_p
    lib.oracle_philox4x32_10.argtypes = [vp, vp, vp]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_noise_bits.argtypes = [c_u64, c_i64, c_i64]
    lib.oracle_noise_bits.restype = ctypes.c_uint32
    lib.oracle_uniform.argtypes = [ctypes.c_uint32]
    lib.oracle_uniform.restype = ctypes.c_float
    lib.oracle_gumbel_of_bits.argtypes = [ctypes.c_uint32]
    lib.oracle_gumbel_of_bits.restype = ctypes.c_double
    lib.oracle_philox_gumbel.argtypes = [c_u64, c_i64, c_i64, c_i64, vp, vp]
    lib.oracle_philox_gumbel.restype = None
    lib.oracle_f32_to_bf16_bits.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_bits.restype = ctypes.c_uint16
    lib.oracle_f32_to_f16_bits.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16_bits.restype = ctypes.c_uint16
    lib.oracle_row_stats.argtypes = [vp, c_i64, c_i64, c_i64, vp, c_i64, c_u64,
                                     c_i64, c_i64, vp, vp, vp, vp, ctypes.c_int,
                                     vp, c_i64, vp, vp]
    lib.oracle_row_stats.restype = ctypes.c_int
    lib.oracle_topk_logprobs.argtypes = [vp, c_i64, c_i64, c_i64, vp, c_i64, vp,
                                         c_i32, c_i64, c_i64, vp, vp]
    lib.oracle_topk_logprobs.restype = ctypes.c_int
    lib.oracle_row_stats_rows.argtypes = [vp, vp, vp, c_i64, c_i64, c_u64, vp, vp, vp, vp,
                                          ctypes.c_int, vp, vp, vp]
    lib.oracle_row_stats_rows.restype = ctypes.c_int
    lib.oracle_topk_rows.argtypes = [vp, vp, c_i64, c_i64, c_i32, vp, vp]
    lib.oracle_topk_rows.restype = ctypes.c_int
    lib.oracle_stash.argtypes = [vp, c_i64, c_i64, c_i64, c_i64, vp, vp, vp, vp, vp, c_i32,
                                 vp, vp, c_i64, c_i32, ctypes.c_int, vp, vp, vp]
    lib.oracle_stash.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _logits_view(logits: np.ndarray):
    """(array, rows, vocab, row_stride) for a 2-D fp32 array whose last axis
    is contiguous (a column slice of a wider buffer is allowed)."""
    assert logits.dtype == np.float32 and logits.ndim == 2
    assert logits.strides[1] == 4, "columns must be contiguous"
    rows, vocab = logits.shape
    stride = logits.strides[0] // 4 if rows > 1 else vocab
    return rows, vocab, stride


def _split(rows_sel, threads):
    threads = max(1, min(threads, len(rows_sel)))
    return [rows_sel[k::threads] for k in range(threads)] if rows_sel else []


# ------------------------------------------------------------------ Philox

def philox4x32_10(ctr, key) -> list[int]:
    """One Philox4x32-10 block: 4 counter words, 2 key words -> 4 words."""
    lib = _load()
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return [int(v) for v in out]


def noise_bits(seed: int, row: int, col: int) -> int:
    return int(_load().oracle_noise_bits(seed, row, col))


def uniform(bits: int) -> float:
    return float(_load().oracle_uniform(bits))


def gumbel_of_bits(bits: int) -> float:
    return float(_load().oracle_gumbel_of_bits(bits))


def philox_gumbel(seed: int, row0: int, rows: int, vocab: int):
    """(bits uint32 [rows, vocab], gumbel float64 [rows, vocab])."""
    lib = _load()
    bits = np.zeros((rows, vocab), dtype=np.uint32)
    g = np.zeros((rows, vocab), dtype=np.float64)
    lib.oracle_philox_gumbel(seed, row0, rows, vocab, _ptr(bits), _ptr(g))
    return bits, g


def f32_to_bf16_bits(x: float) -> int:
    return int(_load().oracle_f32_to_bf16_bits(x))


def f32_to_f16_bits(x: float) -> int:
    return int(_load().oracle_f32_to_f16_bits(x))


# --------------------------------------------------------------- row stats

def row_stats(logits: np.ndarray, temps: np.ndarray, canvas_len: int, seed: int,
              probs_dtype: int = PROBS_NONE, rows_sel=None, threads: int = 1):
    """Oracle row statistics.

    ``logits`` is a 2-D fp32 array (row stride may exceed the vocab). Only
    the rows in ``rows_sel`` (default: all) are computed; the others hold
    -1 / NaN. Returns a dict with ``argmax`` and ``sample`` (int64 [rows]),
    ``entropy`` and ``entropy_check`` (float64 [rows]), ``sample_gap``
    and ``sample_best`` (float64 [rows]: best minus second-best noisy score,
    and the best score) and ``probs`` (uint16 codes [rows, vocab] or None).
    """
    lib = _load()
    rows, vocab, stride = _logits_view(logits)
    temps = np.ascontiguousarray(temps, dtype=np.float32)
    assert temps.size * canvas_len >= rows
    argmax = np.full(rows, -1, dtype=np.int64)
    sample = np.full(rows, -1, dtype=np.int64)
    entropy = np.full(rows, np.nan, dtype=np.float64)
    entropy_check = np.full(rows, np.nan, dtype=np.float64)
    gap = np.full(rows, np.nan, dtype=np.float64)
    best = np.full(rows, np.nan, dtype=np.float64)
    probs = (np.zeros((rows, vocab), dtype=np.uint16)
             if probs_dtype != PROBS_NONE else None)
    rows_sel = list(range(rows)) if rows_sel is None else sorted(int(r) for r in rows_sel)

    def run(part):
        for r in part:
            rc = lib.oracle_row_stats(_ptr(logits), rows, vocab, stride, _ptr(temps),
                                      canvas_len, seed, r, r + 1, _ptr(argmax),
                                      _ptr(sample), _ptr(entropy), _ptr(entropy_check),
                                      probs_dtype, _ptr(probs), vocab, _ptr(gap),
                                      _ptr(best))
            if rc != 0:
                raise MemoryError("oracle_row_stats")

    parts = _split(rows_sel, threads)
    if len(parts) <= 1:
        for p in parts:
            run(p)
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return {"argmax": argmax, "sample": sample, "entropy": entropy,
            "entropy_check": entropy_check, "sample_gap": gap, "sample_best": best,
            "probs": probs}


def topk_logprobs(logits: np.ndarray, temps: np.ndarray, canvas_len: int,
                  keep: np.ndarray, k: int, rows_sel=None, threads: int = 1):
    """Oracle top-k logprobs of the kept rows: (ids int32 [rows, k],
    logprobs float64 [rows, k]); rows not computed hold -1 / NaN."""
    lib = _load()
    rows, vocab, stride = _logits_view(logits)
    temps = np.ascontiguousarray(temps, dtype=np.float32)
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    ids = np.full((rows, max(k, 0)), -1, dtype=np.int32)
    lps = np.full((rows, max(k, 0)), np.nan, dtype=np.float64)
    rows_sel = list(range(rows)) if rows_sel is None else sorted(int(r) for r in rows_sel)

    def run(part):
        for r in part:
            rc = lib.oracle_topk_logprobs(_ptr(logits), rows, vocab, stride, _ptr(temps),
                                          canvas_len, _ptr(keep), k, r, r + 1,
                                          _ptr(ids), _ptr(lps))
            if rc != 0:
                raise MemoryError("oracle_topk_logprobs")

    parts = _split(rows_sel, threads)
    if len(parts) <= 1:
        for p in parts:
            run(p)
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return ids, lps


def _row_pointers(x: np.ndarray):
    assert x.dtype == np.float32 and x.ndim == 2 and x.strides[1] == 4
    base = x.ctypes.data
    return np.array([base + t * x.strides[0] for t in range(x.shape[0])], dtype=np.uint64)


def row_stats_rows(x: np.ndarray, row_ids, temps, seed: int,
                   probs_dtype: int = PROBS_NONE, threads: int = 1):
    """Oracle row statistics of rows given one by one.

    ``x`` is [n, vocab] fp32: row t of it is global row ``row_ids[t]`` (the
    index that keys the noise) with temperature ``temps[t]``. Returns the
    same dict as ``row_stats``, indexed by t.
    """
    lib = _load()
    n, vocab = x.shape
    row_ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    temps = np.ascontiguousarray(temps, dtype=np.float32)
    assert row_ids.size == n and temps.size == n
    out = {"argmax": np.full(n, -1, np.int64), "sample": np.full(n, -1, np.int64),
           "entropy": np.full(n, np.nan), "entropy_check": np.full(n, np.nan),
           "sample_gap": np.full(n, np.nan), "sample_best": np.full(n, np.nan),
           "probs": (np.zeros((n, vocab), np.uint16) if probs_dtype != PROBS_NONE else None)}
    ptrs = _row_pointers(x)

    def run(part):
        for t in part:
            def at(a, w=1):
                return None if a is None else ctypes.c_void_p(a.ctypes.data + t * a.strides[0])
            rc = lib.oracle_row_stats_rows(at(ptrs), at(row_ids), at(temps), 1, vocab, seed,
                                           at(out["argmax"]), at(out["sample"]),
                                           at(out["entropy"]), at(out["entropy_check"]),
                                           probs_dtype, at(out["probs"]), at(out["sample_gap"]),
                                           at(out["sample_best"]))
            if rc != 0:
                raise MemoryError("oracle_row_stats_rows")

    parts = _split(list(range(n)), threads)
    if len(parts) <= 1:
        for part in parts:
            run(part)
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return out


def topk_rows(x: np.ndarray, temps, k: int, threads: int = 1):
    """Oracle top-k of rows given one by one (all treated as kept):
    (ids int32 [n, k], logprobs float64 [n, k])."""
    lib = _load()
    n, vocab = x.shape
    temps = np.ascontiguousarray(temps, dtype=np.float32)
    ids = np.full((n, k), -1, np.int32)
    lps = np.full((n, k), np.nan)
    ptrs = _row_pointers(x)

    def run(part):
        for t in part:
            rc = lib.oracle_topk_rows(ctypes.c_void_p(ptrs.ctypes.data + 8 * t),
                                      ctypes.c_void_p(temps.ctypes.data + 4 * t), 1, vocab, k,
                                      ctypes.c_void_p(ids.ctypes.data + ids.strides[0] * t),
                                      ctypes.c_void_p(lps.ctypes.data + lps.strides[0] * t))
            if rc != 0:
                raise MemoryError("oracle_topk_rows")

    parts = _split(list(range(n)), threads)
    if len(parts) <= 1:
        for part in parts:
            run(part)
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return ids, lps


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))


def stash(logits: np.ndarray, canvas_len: int, src, slots, keep, valid, temps,
          num_topk: int, num_token_ids, token_ids, out_slots: int, width: int,
          logits_mode: bool = False):
    """Oracle stash (see oracle_stash in drs_oracle.c): (ids int32 [out_slots,
    canvas_len, width], values float64 [same], ranks int32 [out_slots,
    canvas_len]). Entries the stash does not write hold -1, NaN and -1.
    token_ids: None, or int32 [m, n] (n >= max num_token_ids)."""
    lib = _load()
    rows, vocab, stride = _logits_view(logits)
    i32 = lambda a: np.ascontiguousarray(a, dtype=np.int32)
    src, slots, valid = i32(src), i32(slots), i32(valid)
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    temps = np.ascontiguousarray(temps, dtype=np.float32)
    m = src.shape[0]
    nti = i32(num_token_ids) if num_token_ids is not None else None
    tid = i32(token_ids) if token_ids is not None else None
    ids_stride = tid.shape[1] if tid is not None else 0
    ids = np.full((out_slots, canvas_len, width), -1, dtype=np.int32)
    vals = np.full((out_slots, canvas_len, width), np.nan, dtype=np.float64)
    ranks = np.full((out_slots, canvas_len), -1, dtype=np.int32)
    rc = lib.oracle_stash(_ptr(logits), stride, vocab, canvas_len, m, _ptr(src), _ptr(slots),
                          _ptr(keep), _ptr(valid), _ptr(temps), num_topk, _ptr(nti), _ptr(tid),
                          ids_stride, width, 1 if logits_mode else 0, _ptr(ids), _ptr(vals),
                          _ptr(ranks))
    if rc != 0:
        raise MemoryError("oracle_stash")
    return ids, vals, ranks
