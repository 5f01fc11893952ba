"""The C ABI library on the host (no GPU needed): it builds for sm_103a,
loads, exports every entry point include/drs.h declares, and its host-side
argument checks reject bad calls before touching the device. The calls here
pass made-up device addresses that are never dereferenced: validation
returns first.
"""
import ctypes
import os
import re

import pytest

import vocab_row_sampling_gb300 as drs
from vocab_row_sampling_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x7F0000000000          # a 256-byte aligned address; never dereferenced
INV, UNS, OK = drs.DRS_ERR_INVALID_ARG, drs.DRS_ERR_UNSUPPORTED, drs.DRS_OK


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return drs.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "drs.h")).read()
    return sorted(set(re.findall(r"\b(drs_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert _declared() == sorted(drs.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in [(0, "DRS_OK"), (-1, "DRS_ERR_INVALID_ARG"), (-2, "DRS_ERR_UNSUPPORTED"),
                       (-3, "DRS_ERR_CUDA"), (-4, "DRS_ERR_DEVICE_TIMEOUT")]:
        assert drs.status_string(code) == name


def test_workspace_sizes(lib):
    assert drs.drs_row_stats_workspace_bytes(2048, 262144) >= 152 * 4 * 32
    assert drs.drs_topk_workspace_bytes(2048, 262144, 0) == 0
    assert drs.drs_topk_workspace_bytes(2048, 262144, 64) >= 152 * 4 * (32 + 64 * 8)


def test_header_sizes_match_the_library(lib):
    """The workspace per row and the no-alloc batch that include/drs.h
    states for rows of 262144 columns are the ones the library computes."""
    with open(os.path.join(_build.INCLUDE, "drs.h")) as f:
        text = " ".join(f.read().split())
    per_row = drs.drs_row_stats_workspace_bytes(2048, 262144) / 2048 / 1024
    stated = float(re.search(r"about ([0-9.]+) KiB per row \* of 262144 columns", text).group(1))
    assert abs(stated - per_row) < 0.1
    fits = max(n for n in range(1, 1024) if drs.drs_row_stats_workspace_bytes(n, 262144) <= 640 * 1024)
    assert int(re.search(r"at most ([0-9]+) rows of 262144 \* columns per batch", text).group(1)) == fits


def _row_stats(lib, rows=4, vocab=16, stride=16, temps=FAKE, canvas=1, row0=0, logits=FAKE,
               outs=FAKE, probs_dtype=1, probs=FAKE, pstride=16, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = drs.drs_row_stats_workspace_bytes(rows, vocab)
    return lib.drs_row_stats(logits, rows, vocab, stride, temps, canvas, 0, row0, outs, outs,
                             outs, probs_dtype, probs, pstride, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,expect", [
    ({"rows": -1}, INV), ({"vocab": 0}, INV), ({"stride": 8}, INV), ({"canvas": 0}, INV),
    ({"row0": -1}, INV), ({"logits": None}, INV), ({"temps": None}, INV),
    ({"outs": None}, INV), ({"probs_dtype": 0}, INV), ({"probs": None}, INV),
    ({"probs_dtype": 3}, INV), ({"pstride": 15}, INV), ({"ws": None}, INV),
    ({"ws_bytes": 64}, INV), ({"ws": FAKE + 16}, INV), ({"logits": FAKE + 2}, INV),
    ({"vocab": drs.DRS_MAX_VOCAB + 1, "stride": drs.DRS_MAX_VOCAB + 1,
      "pstride": drs.DRS_MAX_VOCAB + 1}, UNS),
    ({"rows": 0}, OK),
    ({"rows": 0, "probs_dtype": 0, "probs": None}, OK),
])
def test_row_stats_argument_checks(lib, kw, expect):
    assert _row_stats(lib, **kw) == expect


def _topk(lib, rows=8, vocab=16, stride=16, canvas=4, k=4, keep=FAKE, ids=FAKE, ws=FAKE,
          ws_bytes=None, logits=FAKE):
    if ws_bytes is None:
        ws_bytes = drs.drs_topk_workspace_bytes(rows, vocab, k)
    return lib.drs_topk_logprobs(logits, rows, vocab, stride, FAKE, canvas, keep, k, ids, ids,
                                 ws, ws_bytes, None)


@pytest.mark.parametrize("kw,expect", [
    ({"k": -1}, INV), ({"k": 17}, INV), ({"vocab": 2048, "stride": 2048, "k": 1025}, INV),
    ({"rows": 6}, INV), ({"canvas": 0}, INV), ({"keep": None}, INV), ({"ids": None}, INV),
    ({"ws": None}, INV), ({"ws_bytes": 10}, INV), ({"stride": 15}, INV),
    ({"vocab": drs.DRS_MAX_VOCAB + 1, "stride": drs.DRS_MAX_VOCAB + 1}, UNS),
    ({"k": 0, "ws": None, "ws_bytes": 0}, OK), ({"rows": 0}, OK),
])
def test_topk_argument_checks(lib, kw, expect):
    assert _topk(lib, **kw) == expect


def test_philox_argument_checks(lib):
    assert lib.drs_philox_gumbel(0, -1, 4, 4, FAKE, FAKE, None) == INV
    assert lib.drs_philox_gumbel(0, 0, -1, 4, FAKE, FAKE, None) == INV
    assert lib.drs_philox_gumbel(0, 0, 4, 0, FAKE, FAKE, None) == INV
    assert lib.drs_philox_gumbel(0, 0, 0, 4, FAKE, FAKE, None) == OK
    assert lib.drs_philox_gumbel(0, 0, 4, 4, None, None, None) == OK


def test_binding_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    """No silent fallback: a missing libdrs.so raises."""
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(drs, "_lib", None)
    with pytest.raises(RuntimeError):
        drs.load()


def test_scaled_logits_argument_checks(lib):
    assert lib.drs_scaled_logits(FAKE, -1, 1.0, FAKE, None) == INV
    assert lib.drs_scaled_logits(None, 4, 1.0, FAKE, None) == INV
    assert lib.drs_scaled_logits(FAKE, 4, 1.0, FAKE + 2, None) == INV
    assert lib.drs_scaled_logits(FAKE, 0, 1.0, FAKE, None) == OK


def _stash(lib, requests=2, logits_rows=4, vocab=16, stride=16, canvas=2, ptr=FAKE, k=3, nti=None,
           tok=None, ids_stride=0, out_slots=2, width=4, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = drs.drs_stash_workspace_bytes(requests, canvas, vocab, k)
    return lib.drs_stash_converged_logprobs(ptr, logits_rows, vocab, stride, canvas, requests, ptr,
                                            ptr, ptr, ptr, ptr, k, nti, tok, ids_stride, out_slots,
                                            width, ptr, ptr, ptr, 0, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,expect", [
    ({"requests": 0}, OK),                          # nothing to do, nothing launched
    ({"requests": -1}, INV),
    ({"canvas": 0}, INV),
    ({"stride": 8}, INV),
    ({"vocab": 0}, INV),
    ({"vocab": drs.DRS_MAX_VOCAB + 1, "stride": drs.DRS_MAX_VOCAB + 1}, UNS),
    ({"k": -1}, INV),
    ({"k": 17}, INV),                               # more than the vocabulary
    ({"k": 3, "width": 3}, INV),                    # width < num_topk + 1
    ({"width": 0, "k": 0}, INV),
    ({"tok": FAKE, "ids_stride": 4}, INV),          # token ids without their counts
    ({"tok": FAKE, "nti": FAKE, "ids_stride": 0}, INV),
    ({"ptr": 0}, INV),
    ({"ws": 0}, INV),
    ({"ws_bytes": 16}, INV),
    ({"ws": FAKE + 8}, INV),
])
def test_stash_argument_checks(lib, kw, expect):
    assert _stash(lib, **kw) == expect


def test_stash_workspace_sizes(lib):
    assert drs.drs_stash_workspace_bytes(8, 256, 262144, 20) >= 8 * 256 * 20 * 8
    assert drs.drs_stash_workspace_bytes(8, 256, 262144, 1025) == 0
    assert drs.drs_stash_workspace_bytes(-1, 256, 262144, 20) == 0


def test_split_plan_argument_checks(lib):
    out = [ctypes.c_int64(7), ctypes.c_int32(7), ctypes.c_int32(7), ctypes.c_int32(7)]
    refs = [ctypes.byref(o) for o in out]
    assert lib.drs_row_split_plan(2048, 262144, 20, 1, 1, 1, None, *refs[1:]) == INV
    assert lib.drs_row_split_plan(-1, 262144, 20, 1, 1, 1, *refs) == INV
    assert lib.drs_row_split_plan(2048, 0, 20, 1, 1, 1, *refs) == INV
    assert lib.drs_row_split_plan(2048, 262144, 20, 0, 1, 1, *refs) == INV
    assert lib.drs_row_split_plan(2048, 262144, 20, 1, 3, 1, *refs) == INV
    # zero rows: nothing to divide
    assert lib.drs_row_split_plan(0, 262144, 20, 1, 1, 0, *refs) == OK
    assert [o.value for o in out] == [0, 0, 0, 0]
    # several seeds always take the two passes alone
    assert lib.drs_row_split_plan(2048, 262144, 0, 8, 0, 1, *refs) == OK
    assert [o.value for o in out] == [0, 0, 0, 0]
