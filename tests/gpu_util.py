"""Helpers shared by the GPU parity tests: run the CUDA library through its
C ABI binding and bring results back as numpy; run the oracle on the same
bytes."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

TORCH_PROBS = {0: None, 1: torch.bfloat16, 2: torch.float16}
THREADS = max(1, min(32, os.cpu_count() or 1))


def drs():
    import vocab_row_sampling_gb300 as lib
    lib.load(build_if_missing=True)
    return lib


def gpu_row_stats(logits, temps, canvas_len, seed, probs_dtype, row0=0):
    """logits: CUDA [rows, vocab] view (any row stride). Returns numpy dict."""
    lib = drs()
    a, s, e, p = lib.row_stats(logits, temps, canvas_len, seed, TORCH_PROBS[probs_dtype], row0=row0)
    torch.cuda.synchronize()
    assert lib.drs_get_device_error() == 0
    out = {"argmax": a.cpu().numpy(), "sample": s.cpu().numpy(), "entropy": e.cpu().numpy(),
           "probs": None}
    if p is not None:
        out["probs"] = p.view(torch.int16).cpu().numpy().view(np.uint16)
    return out


def oracle_rows(logits, temps_cpu, canvas_len, seed, probs_dtype, rows_sel, row0=0):
    """Oracle on the given rows of a (CUDA or CPU) logits view."""
    rows_sel = np.asarray(rows_sel, dtype=np.int64)
    x = logits[torch.as_tensor(rows_sel, device=logits.device)].cpu().numpy()
    x = np.ascontiguousarray(x, dtype=np.float32)
    gids = rows_sel + row0
    temps = np.asarray(temps_cpu, dtype=np.float32)[gids // canvas_len]
    return oracle.row_stats_rows(x, gids, temps, seed, probs_dtype, threads=THREADS)


def subset(d, rows_sel):
    rows_sel = np.asarray(rows_sel, dtype=np.int64)
    return {k: (None if v is None else v[rows_sel]) for k, v in d.items()}


def sample_rows(rows, n, seed=0, always=()):
    rng = np.random.default_rng(seed)
    pick = set(int(r) for r in always if 0 <= r < rows)
    pick.update(int(r) for r in rng.choice(rows, size=min(n, rows), replace=False))
    return np.array(sorted(pick), dtype=np.int64)
