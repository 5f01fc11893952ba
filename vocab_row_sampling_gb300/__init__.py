"""GB300-native DiffusionGemma per-row sampler statistics.

A thin ctypes binding of ``libdrs.so`` (declared in ``include/drs.h``). Every
function here only marshals arguments: pointers of torch tensors, sizes, the
current CUDA stream. All of the arithmetic runs in the library's CUDA kernels;
there is no CPU fallback. Importing the package works without a GPU; calling
into the library needs the built ``libdrs.so`` and a CUDA device, and raises
otherwise.

Entry points (same names as the C ABI):
  drs_row_stats, drs_row_stats_workspace_bytes, drs_row_stats_noalloc,
  drs_row_stats_topk, drs_row_stats_topk_workspace_bytes, drs_topk_logprobs,
  drs_topk_workspace_bytes, drs_philox_gumbel, drs_scaled_logits,
  drs_stash_converged_logprobs, drs_stash_workspace_bytes,
  drs_status_string, drs_get_device_error.
Convenience wrappers that allocate outputs: row_stats, row_stats_topk,
topk_logprobs, philox_gumbel, stash_converged_logprobs.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

DRS_OK = 0
DRS_ERR_INVALID_ARG = -1
DRS_ERR_UNSUPPORTED = -2
DRS_ERR_CUDA = -3
DRS_ERR_DEVICE_TIMEOUT = -4

DRS_PROBS_NONE, DRS_PROBS_BF16, DRS_PROBS_FP16 = 0, 1, 2
DRS_MAX_VOCAB = 2097152

EXPORTED = ("drs_row_stats", "drs_row_stats_workspace_bytes", "drs_row_stats_noalloc",
            "drs_row_stats_topk", "drs_row_stats_topk_workspace_bytes", "drs_topk_logprobs",
            "drs_topk_workspace_bytes", "drs_philox_gumbel", "drs_scaled_logits",
            "drs_status_string", "drs_get_device_error", "drs_test_inject_fault",
            "drs_kernel_timing", "drs_kernel_times", "drs_row_stats_seeds",
            "drs_row_stats_seeds_workspace_bytes", "drs_stash_converged_logprobs",
            "drs_stash_workspace_bytes", "drs_test_two_pass",
            "drs_row_split_plan")


class DrsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libdrs.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libdrs.so is not built ({path}); run "
                               "vocab_row_sampling_gb300._build.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    i64, u64, i32, vp, sz = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32,
                             ctypes.c_void_p, ctypes.c_size_t)
    lib.drs_row_stats_workspace_bytes.argtypes = [i64, i64]
    lib.drs_row_stats_workspace_bytes.restype = sz
    lib.drs_row_stats.argtypes = [vp, i64, i64, i64, vp, i64, u64, i64, vp, vp, vp,
                                  ctypes.c_int, vp, i64, vp, sz, vp]
    lib.drs_row_stats.restype = ctypes.c_int
    lib.drs_row_stats_noalloc.argtypes = [vp, i64, i64, i64, vp, i64, u64, i64, vp, vp, vp,
                                          ctypes.c_int, vp, i64, vp]
    lib.drs_row_stats_noalloc.restype = ctypes.c_int
    lib.drs_row_stats_topk_workspace_bytes.argtypes = [i64, i64, i32]
    lib.drs_row_stats_topk_workspace_bytes.restype = sz
    lib.drs_row_stats_topk.argtypes = [vp, i64, i64, i64, vp, i64, u64, i64, vp, vp, vp,
                                       ctypes.c_int, vp, i64, vp, i32, vp, vp, vp, sz, vp]
    lib.drs_row_stats_topk.restype = ctypes.c_int
    lib.drs_topk_workspace_bytes.argtypes = [i64, i64, i32]
    lib.drs_topk_workspace_bytes.restype = sz
    lib.drs_topk_logprobs.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, vp, vp, vp, sz, vp]
    lib.drs_topk_logprobs.restype = ctypes.c_int
    lib.drs_stash_workspace_bytes.argtypes = [i64, i64, i64, i32]
    lib.drs_stash_workspace_bytes.restype = sz
    lib.drs_stash_converged_logprobs.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                                                 i32, vp, vp, i64, i64, i32, vp, vp, vp,
                                                 ctypes.c_int, vp, sz, vp]
    lib.drs_stash_converged_logprobs.restype = ctypes.c_int
    lib.drs_philox_gumbel.argtypes = [u64, i64, i64, i64, vp, vp, vp]
    lib.drs_philox_gumbel.restype = ctypes.c_int
    lib.drs_scaled_logits.argtypes = [vp, i64, ctypes.c_float, vp, vp]
    lib.drs_scaled_logits.restype = ctypes.c_int
    lib.drs_status_string.argtypes = [ctypes.c_int]
    lib.drs_status_string.restype = ctypes.c_char_p
    lib.drs_test_inject_fault.argtypes = [ctypes.c_int]
    lib.drs_test_inject_fault.restype = None
    lib.drs_test_two_pass.argtypes = [ctypes.c_int]
    lib.drs_test_two_pass.restype = None
    lib.drs_row_split_plan.argtypes = [i64, i64, i32, i32, ctypes.c_int, i32, vp, vp, vp, vp]
    lib.drs_row_split_plan.restype = ctypes.c_int
    lib.drs_get_device_error.argtypes = [vp]
    lib.drs_get_device_error.restype = ctypes.c_int
    lib.drs_row_stats_seeds_workspace_bytes.argtypes = [i64, i64, i32]
    lib.drs_row_stats_seeds_workspace_bytes.restype = sz
    lib.drs_row_stats_seeds.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, i64, vp, vp, vp,
                                        ctypes.c_int, vp, i64, vp, sz, vp]
    lib.drs_row_stats_seeds.restype = ctypes.c_int
    lib.drs_kernel_timing.argtypes = [ctypes.c_int]
    lib.drs_kernel_timing.restype = ctypes.c_int
    lib.drs_kernel_times.argtypes = [vp, i32, vp]
    lib.drs_kernel_times.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().drs_status_string(status).decode()


drs_status_string = status_string


def _check(status: int, what: str):
    if status != DRS_OK:
        raise DrsError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _row_stride(logits) -> int:
    assert logits.dim() == 2 and logits.stride(1) == 1, "logits: 2-D, unit column stride"
    return logits.stride(0) if logits.shape[0] > 1 else max(logits.shape[1], logits.stride(0))


# ------------------------------------------------------------- raw entry points

def drs_row_stats_workspace_bytes(rows: int, vocab: int) -> int:
    return int(load().drs_row_stats_workspace_bytes(rows, vocab))


def drs_row_stats(logits, temps, canvas_len, seed, argmax, sample, entropy,
                  probs_dtype=DRS_PROBS_NONE, probs=None, workspace=None, stream=None,
                  row0=0):
    """Launch drs_row_stats on torch CUDA tensors (outputs preallocated)."""
    rows, vocab = logits.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    pstride = 0 if probs is None else probs.stride(0)
    st = load().drs_row_stats(_ptr(logits), rows, vocab, _row_stride(logits), _ptr(temps),
                              canvas_len, seed & (2**64 - 1), row0, _ptr(argmax), _ptr(sample),
                              _ptr(entropy), probs_dtype, _ptr(probs), pstride,
                              _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "drs_row_stats")


def drs_row_stats_noalloc(logits, temps, canvas_len, seed, argmax, sample, entropy,
                          probs_dtype=DRS_PROBS_NONE, probs=None, stream=None, row0=0):
    """drs_row_stats with the library's fixed device workspace: for callers
    that cannot allocate device memory (see include/drs.h). Calls that can
    overlap on the GPU share that workspace and race."""
    rows, vocab = logits.shape
    pstride = 0 if probs is None else probs.stride(0)
    st = load().drs_row_stats_noalloc(_ptr(logits), rows, vocab, _row_stride(logits),
                                      _ptr(temps), canvas_len, seed & (2**64 - 1), row0,
                                      _ptr(argmax), _ptr(sample), _ptr(entropy), probs_dtype,
                                      _ptr(probs), pstride, _stream(stream))
    _check(st, "drs_row_stats_noalloc")


def drs_row_stats_seeds_workspace_bytes(rows: int, vocab: int, n_seeds: int) -> int:
    return int(load().drs_row_stats_seeds_workspace_bytes(rows, vocab, n_seeds))


def drs_row_stats_seeds(logits, temps, canvas_len, seeds, argmax, samples, entropy,
                        probs_dtype=DRS_PROBS_NONE, probs=None, workspace=None, stream=None,
                        row0=0):
    """Launch drs_row_stats_seeds: `seeds` a sequence of ints (host), samples
    an int64 CUDA tensor [len(seeds), rows]."""
    rows, vocab = logits.shape
    n = len(seeds)
    keys = (ctypes.c_uint64 * max(n, 1))(*[int(x) & (2**64 - 1) for x in seeds])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    pstride = 0 if probs is None else probs.stride(0)
    st = load().drs_row_stats_seeds(_ptr(logits), rows, vocab, _row_stride(logits), _ptr(temps),
                                    canvas_len, ctypes.cast(keys, ctypes.c_void_p), n, row0,
                                    _ptr(argmax), _ptr(samples), _ptr(entropy), probs_dtype,
                                    _ptr(probs), pstride, _ptr(workspace), ws_bytes,
                                    _stream(stream))
    _check(st, "drs_row_stats_seeds")


def drs_row_stats_topk_workspace_bytes(rows: int, vocab: int, k: int) -> int:
    return int(load().drs_row_stats_topk_workspace_bytes(rows, vocab, k))


def drs_row_stats_topk(logits, temps, canvas_len, seed, argmax, sample, entropy, probs_dtype,
                       probs, keep, k, out_ids, out_logprobs, workspace=None, stream=None, row0=0):
    """Launch drs_row_stats_topk (row statistics and the top-k logprobs of
    converged rows, one read of the logits) on torch CUDA tensors."""
    rows, vocab = logits.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    pstride = 0 if probs is None else probs.stride(0)
    st = load().drs_row_stats_topk(_ptr(logits), rows, vocab, _row_stride(logits), _ptr(temps),
                                   canvas_len, seed & (2**64 - 1), row0, _ptr(argmax),
                                   _ptr(sample), _ptr(entropy), probs_dtype, _ptr(probs), pstride,
                                   _ptr(keep), k, _ptr(out_ids), _ptr(out_logprobs),
                                   _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "drs_row_stats_topk")


def drs_topk_workspace_bytes(rows: int, vocab: int, k: int) -> int:
    return int(load().drs_topk_workspace_bytes(rows, vocab, k))


def drs_topk_logprobs(logits, temps, canvas_len, keep, k, out_ids, out_logprobs,
                      workspace=None, stream=None):
    rows, vocab = logits.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().drs_topk_logprobs(_ptr(logits), rows, vocab, _row_stride(logits), _ptr(temps),
                                  canvas_len, _ptr(keep), k, _ptr(out_ids), _ptr(out_logprobs),
                                  _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "drs_topk_logprobs")


def drs_stash_workspace_bytes(requests: int, canvas_len: int, vocab: int, num_topk: int) -> int:
    return load().drs_stash_workspace_bytes(requests, canvas_len, vocab, num_topk)


def drs_stash_converged_logprobs(logits, canvas_len, src, slots, keep, valid, temps, num_topk,
                                 num_token_ids, token_ids, out_ids, out_logprobs, out_ranks,
                                 logits_mode, workspace=None, stream=None):
    """out_ids / out_logprobs: [out_slots, canvas_len, width]; out_ranks:
    [out_slots, canvas_len]; token_ids: None or int32 [requests, n]."""
    rows, vocab = logits.shape
    requests = src.shape[0]
    out_slots, _, width = out_ids.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ids_stride = token_ids.stride(0) if token_ids is not None else 0
    st = load().drs_stash_converged_logprobs(
        _ptr(logits), rows, vocab, _row_stride(logits), canvas_len, requests, _ptr(src),
        _ptr(slots), _ptr(keep), _ptr(valid), _ptr(temps), num_topk, _ptr(num_token_ids),
        _ptr(token_ids), ids_stride, out_slots, width, _ptr(out_ids), _ptr(out_logprobs),
        _ptr(out_ranks), 1 if logits_mode else 0, _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "drs_stash_converged_logprobs")


def drs_philox_gumbel(seed, row0, rows, vocab, out_bits=None, out_gumbel=None, stream=None):
    st = load().drs_philox_gumbel(seed & (2**64 - 1), row0, rows, vocab, _ptr(out_bits),
                                  _ptr(out_gumbel), _stream(stream))
    _check(st, "drs_philox_gumbel")


def drs_scaled_logits(logits, temp: float, out, stream=None):
    """out = logits / max(temp, 1e-10) elementwise (contiguous fp32 tensors)."""
    assert logits.is_contiguous() and out.is_contiguous() and out.numel() == logits.numel()
    st = load().drs_scaled_logits(_ptr(logits), logits.numel(), temp, _ptr(out), _stream(stream))
    _check(st, "drs_scaled_logits")


KERNEL_NAMES = ("split_prep", "split_pass1", "split_merge", "split_pass2", "split_cluster",
                "split_finish")


def drs_kernel_timing(enable: bool) -> None:
    """Measurement hook: record CUDA events around the row kernels of every
    following call on the current device (see include/drs.h)."""
    _check(load().drs_kernel_timing(1 if enable else 0), "drs_kernel_timing")


def drs_kernel_times():
    """Average ms of each row kernel over the calls recorded since timing was
    switched on: ({kernel name: ms}, number of calls averaged)."""
    out = (ctypes.c_float * len(KERNEL_NAMES))()
    calls = ctypes.c_int32(0)
    _check(load().drs_kernel_times(ctypes.cast(out, ctypes.c_void_p), len(KERNEL_NAMES),
                                   ctypes.cast(ctypes.pointer(calls), ctypes.c_void_p)),
           "drs_kernel_times")
    return dict(zip(KERNEL_NAMES, (float(v) for v in out))), int(calls.value)


def drs_test_inject_fault(code: int) -> None:
    """Test hook: in the next row-statistics call a CTA never fills its first
    stage, so that the bounded waits on it run out (see include/drs.h)."""
    load().drs_test_inject_fault(code)


def drs_test_two_pass(on: bool) -> None:
    """Test hook: every following row-statistics call takes the two passes
    over the logits instead of the one-read cluster kernel (see
    include/drs.h)."""
    load().drs_test_two_pass(1 if on else 0)


def cluster_rows(rows: int, vocab: int, k: int, n_seeds: int = 1, probs_dtype: int = DRS_PROBS_BF16,
                 stats: bool = True):
    """How a row-statistics call of these sizes shares its rows on the
    current device (drs_row_split_plan): None when it takes the two passes
    alone, else a dict with the rows of the cluster kernel ("head"), of the
    two passes beside it ("tail"), the cluster size, the clusters resident
    at once and the SMs they leave free."""
    head, size, ncl, free = ctypes.c_int64(0), ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load().drs_row_split_plan(rows, vocab, k, n_seeds, probs_dtype, 1 if stats else 0,
                                     ctypes.byref(head), ctypes.byref(size), ctypes.byref(ncl),
                                     ctypes.byref(free)), "drs_row_split_plan")
    if size.value == 0:
        return None
    return {"head": int(head.value), "tail": int(rows - head.value), "cluster_size": int(size.value),
            "clusters": int(ncl.value), "free_sms": int(free.value)}


def drs_get_device_error(stream=None) -> int:
    return int(load().drs_get_device_error(_stream(stream)))


# ------------------------------------------------------------- conveniences

_workspaces = {}


def workspace(nbytes: int, device):
    """A cached device workspace of at least nbytes (256-byte aligned)."""
    import torch
    key = (str(device), nbytes)
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def row_stats(logits, temps, canvas_len: int, seed: int, probs_dtype=None, stream=None,
              row0: int = 0):
    """Allocate outputs and run drs_row_stats; returns (argmax, sample,
    entropy, probs) like the page's sample_row_stats."""
    import torch
    rows, vocab = logits.shape
    dev = logits.device
    argmax = torch.empty(rows, dtype=torch.int64, device=dev)
    sample = torch.empty(rows, dtype=torch.int64, device=dev)
    entropy = torch.empty(rows, dtype=torch.float32, device=dev)
    code = {None: DRS_PROBS_NONE, torch.bfloat16: DRS_PROBS_BF16,
            torch.float16: DRS_PROBS_FP16}[probs_dtype]
    probs = None if probs_dtype is None else torch.empty(rows, vocab, dtype=probs_dtype, device=dev)
    if rows == 0:
        return argmax, sample, entropy, probs
    ws = workspace(drs_row_stats_workspace_bytes(rows, vocab), dev)
    drs_row_stats(logits, temps, canvas_len, seed, argmax, sample, entropy, code, probs, ws,
                  stream, row0)
    return argmax, sample, entropy, probs


def row_stats_seeds(logits, temps, canvas_len: int, seeds, probs_dtype=None, stream=None,
                    row0: int = 0):
    """Allocate outputs and run drs_row_stats_seeds; returns (argmax,
    samples [len(seeds), rows], entropy, probs)."""
    import torch
    rows, vocab = logits.shape
    dev = logits.device
    argmax = torch.empty(rows, dtype=torch.int64, device=dev)
    samples = torch.empty(len(seeds), rows, dtype=torch.int64, device=dev)
    entropy = torch.empty(rows, dtype=torch.float32, device=dev)
    code = {None: DRS_PROBS_NONE, torch.bfloat16: DRS_PROBS_BF16,
            torch.float16: DRS_PROBS_FP16}[probs_dtype]
    probs = None if probs_dtype is None else torch.empty(rows, vocab, dtype=probs_dtype, device=dev)
    if rows == 0:
        return argmax, samples, entropy, probs
    ws = workspace(drs_row_stats_seeds_workspace_bytes(rows, vocab, len(seeds)), dev)
    drs_row_stats_seeds(logits, temps, canvas_len, seeds, argmax, samples, entropy, code, probs,
                        ws, stream, row0)
    return argmax, samples, entropy, probs


def row_stats_topk(logits, temps, canvas_len: int, seed: int, keep, k: int, probs_dtype=None,
                   out_ids=None, out_logprobs=None, stream=None, row0: int = 0):
    """Allocate outputs and run drs_row_stats_topk; returns (argmax, sample,
    entropy, probs, out_ids, out_logprobs). Rows of unconverged slots keep
    the given (or -1 / NaN filled) top-k outputs."""
    import torch
    rows, vocab = logits.shape
    dev = logits.device
    argmax = torch.empty(rows, dtype=torch.int64, device=dev)
    sample = torch.empty(rows, dtype=torch.int64, device=dev)
    entropy = torch.empty(rows, dtype=torch.float32, device=dev)
    code = {None: DRS_PROBS_NONE, torch.bfloat16: DRS_PROBS_BF16,
            torch.float16: DRS_PROBS_FP16}[probs_dtype]
    probs = None if probs_dtype is None else torch.empty(rows, vocab, dtype=probs_dtype, device=dev)
    if out_ids is None:
        out_ids = torch.full((rows, k), -1, dtype=torch.int32, device=dev)
    if out_logprobs is None:
        out_logprobs = torch.full((rows, k), float("nan"), dtype=torch.float32, device=dev)
    if rows == 0:
        return argmax, sample, entropy, probs, out_ids, out_logprobs
    ws = workspace(max(drs_row_stats_topk_workspace_bytes(rows, vocab, k),
                       drs_row_stats_workspace_bytes(rows, vocab)), dev)
    drs_row_stats_topk(logits, temps, canvas_len, seed, argmax, sample, entropy, code, probs,
                       keep, k, out_ids, out_logprobs, ws, stream, row0)
    return argmax, sample, entropy, probs, out_ids, out_logprobs


def topk_logprobs(logits, temps, canvas_len: int, keep, k: int, out_ids=None,
                  out_logprobs=None, stream=None):
    """Top-k ids and logprobs of the rows of kept slots (other rows of the
    given outputs are left as they are)."""
    import torch
    rows, vocab = logits.shape
    dev = logits.device
    if out_ids is None:
        out_ids = torch.full((rows, k), -1, dtype=torch.int32, device=dev)
    if out_logprobs is None:
        out_logprobs = torch.full((rows, k), float("nan"), dtype=torch.float32, device=dev)
    ws = workspace(drs_topk_workspace_bytes(rows, vocab, k), dev)
    drs_topk_logprobs(logits, temps, canvas_len, keep, k, out_ids, out_logprobs, ws, stream)
    return out_ids, out_logprobs


def philox_gumbel(seed: int, row0: int, rows: int, vocab: int, device="cuda", stream=None):
    import torch
    bits = torch.empty(rows, vocab, dtype=torch.int32, device=device)
    g = torch.empty(rows, vocab, dtype=torch.float32, device=device)
    drs_philox_gumbel(seed, row0, rows, vocab, bits, g, stream)
    return bits, g


def stash_converged_logprobs(logits, canvas_len: int, src, slots, keep, valid, temps,
                             num_topk: int, num_token_ids=None, token_ids=None, out_ids=None,
                             out_logprobs=None, out_ranks=None, out_slots: int | None = None,
                             width: int | None = None, logits_mode: bool = False, stream=None):
    """The stash (see drs_stash_converged_logprobs); outputs allocated when
    not given, filled with -1 / NaN / -1 where the stash does not write."""
    import torch
    dev = logits.device
    if out_ids is None:
        out_slots = int(src.shape[0]) if out_slots is None else out_slots
        width = num_topk + 1 if width is None else width
        out_ids = torch.full((out_slots, canvas_len, width), -1, dtype=torch.int32, device=dev)
    if out_logprobs is None:
        out_logprobs = torch.full(out_ids.shape, float("nan"), dtype=torch.float32, device=dev)
    if out_ranks is None:
        out_ranks = torch.full(out_ids.shape[:2], -1, dtype=torch.int32, device=dev)
    ws = workspace(drs_stash_workspace_bytes(int(src.shape[0]), canvas_len, logits.shape[1],
                                             num_topk), dev)
    drs_stash_converged_logprobs(logits, canvas_len, src, slots, keep, valid, temps, num_topk,
                                 num_token_ids, token_ids, out_ids, out_logprobs, out_ranks,
                                 logits_mode, ws, stream)
    return out_ids, out_logprobs, out_ranks
