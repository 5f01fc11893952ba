"""Benchmark of the DiffusionGemma row-statistics hot path on GB300.

One step = one pass of the whole path over one batch: drs_row_stats_topk,
the row statistics (argmax, Gumbel-max sample, entropy, bf16 softmax) of
2048 x 262144 fp32 logits and the top-k logprobs (k = 20) of the rows of the
converged (even) slots. Inputs are synthetic (workloads.py, "step") and
resident in HBM when the timed region starts; at 2.1 GB they are larger than
L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0). `value` is rows/s over all GPUs. `roofline`
describes the dominant kernel, pass 2 (probabilities, Gumbel race, top-k
candidates): its algorithmic bytes (every logit read once, every probability
written once: rows*V*4 + rows*V*2) over its average CUDA-event duration,
the events recorded on the call's stream around each kernel by the
library's measurement hook during a second run of the timed steps (the
events cost about 15 us per call, so the steps whose time gives `value` run
without them; clocks are sampled over both runs). `kernels` gives every
kernel of the call the same way and the whole call, plus the two separate
calls (drs_row_stats, then drs_topk_logprobs) timed briefly; `e2e` repeats
the step through the public API from pinned host buffers, copies included;
`cpu_baseline` times the CPU oracle on a bounded sample of the same rows.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --rows 256 --no-e2e --cpu-seconds 0   (a smaller case of
      the same workload, e.g. for a counter capture; not a headline number)
Under torchrun each rank runs its own batch (weak scaling, rows keyed by
global row index so results equal one big batch); no collective touches
the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "rows/s and achieved HBM GB/s (% of roofline) for row_stats at 2048x262144 fp32"
WORKLOAD = "step"  # set from --workload
WORKLOAD_TEXT = {
    "step": "step: 2048 x 262144 fp32 logits, bf16 probs, top-k 20 on the even (converged) slots",
    "wide": "wide: 512 x 2097152 fp32 logits (the step recipe on rows of 2^21 columns), bf16 "
            "probs, top-k 20 on the even (converged) slots; not the headline workload",
}
FALLBACK_HBM_GBS = 6800.0


def _peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxs.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs),
                "reasons": sorted(reasons), "samples": len(sms)}


def _clocks_rejected(c):
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(c.get("reasons", [])):
        return True
    if c.get("sm_mhz") and c.get("sm_max_mhz") and c["sm_mhz"] < 0.6 * c["sm_max_mhz"]:
        return True
    return False


# ---------------------------------------------------------------- our arm

def _make_batch(rank: int, rows=None):
    w = workloads.make(WORKLOAD, device="cuda", data_seed=rank, rows=rows)
    return w


def shard_layout(rank: int, rows: int, canvas_len: int):
    """Weak scaling: rank r owns global rows [r*rows, (r+1)*rows), whose
    slots start at r*rows/canvas_len. Returns (row0, first_slot)."""
    assert rows % canvas_len == 0
    return rank * rows, rank * rows // canvas_len


def global_temps(temps_local, rank: int, rows: int, canvas_len: int):
    """A per-slot temperature array indexed by global slot in which this
    rank's slots hold its temperatures (the others are never read)."""
    _, slot0 = shard_layout(rank, rows, canvas_len)
    out = torch.zeros(slot0 + temps_local.numel(), dtype=torch.float32,
                      device=temps_local.device)
    out[slot0:] = temps_local
    return out


def global_keep(keep_local, rank: int, rows: int, canvas_len: int):
    """The keep flags indexed by global slot, like global_temps."""
    _, slot0 = shard_layout(rank, rows, canvas_len)
    out = torch.zeros(slot0 + keep_local.numel(), dtype=torch.uint8, device=keep_local.device)
    out[slot0:] = keep_local
    return out


def _run_ours(args, world, rank, local):
    import vocab_row_sampling_gb300 as drs
    drs.load(build_if_missing=True)
    torch.cuda.set_device(local)
    w = _make_batch(rank, args.rows)
    rows, V, stride = w["rows"], w["vocab"], w["row_stride"]
    logits = w["logits"][:, :V]
    temps, keep = w["temps"].cuda(), w["keep"].cuda()
    k = w["k"]
    row0, _ = shard_layout(rank, rows, w["canvas_len"])
    dev = logits.device
    stream = torch.cuda.current_stream()
    temps_all = global_temps(temps, rank, rows, w["canvas_len"])
    keep_all = global_keep(keep, rank, rows, w["canvas_len"])

    argmax = torch.empty(rows, dtype=torch.int64, device=dev)
    sample = torch.empty(rows, dtype=torch.int64, device=dev)
    entropy = torch.empty(rows, dtype=torch.float32, device=dev)
    probs = torch.empty(rows, V, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(rows, k, dtype=torch.int32, device=dev)
    lps = torch.empty(rows, k, dtype=torch.float32, device=dev)
    ws_rs = drs.workspace(drs.drs_row_stats_workspace_bytes(rows, V), dev)
    ws_tk = drs.workspace(drs.drs_topk_workspace_bytes(rows, V, k), dev)
    ws_fused = drs.workspace(drs.drs_row_stats_topk_workspace_bytes(rows, V, k), dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        drs.drs_row_stats_topk(logits, temps_all, w["canvas_len"], 0, argmax, sample, entropy,
                               drs.DRS_PROBS_BF16, probs, keep_all, k, ids, lps, ws_fused,
                               stream, row0=row0)
        if ev is not None:
            ev[1].record(stream)

    # the stash of the converged requests (one per slot: src = slots = the
    # slot, every position valid), top-k + the argmax column
    n_slots = rows // w["canvas_len"]
    req = torch.arange(n_slots, dtype=torch.int32, device=dev)
    valid_all = torch.full((n_slots,), w["canvas_len"], dtype=torch.int32, device=dev)
    st_ids = torch.empty(n_slots, w["canvas_len"], k + 1, dtype=torch.int32, device=dev)
    st_vals = torch.empty(n_slots, w["canvas_len"], k + 1, dtype=torch.float32, device=dev)
    st_ranks = torch.empty(n_slots, w["canvas_len"], dtype=torch.int32, device=dev)
    ws_st = drs.workspace(drs.drs_stash_workspace_bytes(n_slots, w["canvas_len"], V, k), dev)

    def stash_ms(n=3):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        t = []
        for _ in range(n + 1):
            evs[0].record(stream)
            drs.drs_stash_converged_logprobs(logits, w["canvas_len"], req, req, keep, valid_all,
                                             temps, k, None, None, st_ids, st_vals, st_ranks,
                                             False, ws_st, stream)
            evs[1].record(stream)
            torch.cuda.synchronize()
            t.append(evs[0].elapsed_time(evs[1]))
        return sum(t[1:]) / n

    def separate(n=3):
        """The two separate calls, timed briefly (context for the fused one)."""
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        rs, tk = [], []
        for _ in range(n + 1):
            evs[0].record(stream)
            drs.drs_row_stats(logits, temps_all, w["canvas_len"], 0, argmax, sample, entropy,
                              drs.DRS_PROBS_BF16, probs, ws_rs, stream, row0=row0)
            evs[1].record(stream)
            drs.drs_topk_logprobs(logits, temps, w["canvas_len"], keep, k, ids, lps, ws_tk, stream)
            evs[2].record(stream)
            torch.cuda.synchronize()
            rs.append(evs[0].elapsed_time(evs[1]))
            tk.append(evs[1].elapsed_time(evs[2]))
        return sum(rs[1:]) / n, sum(tk[1:]) / n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if drs.drs_get_device_error() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    def timed():
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(torch.cuda.current_device()) as clk:
            start.record(stream)
            for i in range(args.steps):
                step(evs[i])
            stop.record(stream)
            torch.cuda.synchronize()
            # the same steps again with the library's events around each
            # kernel (they cost about 15 us per call, so the steps above run
            # without them)
            drs.drs_kernel_timing(True)
            for i in range(args.steps):
                step()
            torch.cuda.synchronize()
            drs.drs_kernel_timing(False)
        _barrier(world)
        total_ms = start.elapsed_time(stop)
        rs_ms = [e[0].elapsed_time(e[1]) for e in evs]
        return total_ms, rs_ms, clk.summary(), drs.drs_kernel_times()

    total_ms, rs_ms, clocks, ktimes = timed()
    if _clocks_rejected(clocks):
        total_ms, rs_ms, clocks, ktimes = timed()
        clocks["remeasured"] = True
    kernel_ms, kernel_calls = ktimes
    if drs.drs_get_device_error() != 0:
        raise RuntimeError("device-side wait timed out during the timed region")
    total_ms = _max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = world * rows * args.steps / (total_ms / 1e3)

    rs_avg_ms = sum(rs_ms) / len(rs_ms)
    sep_rs_ms, tk_avg_ms = separate()
    stash_avg_ms = stash_ms()
    bytes_rs = rows * V * 4 + rows * V * 2      # each logit read once, each probability written once
    kept_rows = int(keep[: rows // w["canvas_len"]].sum().item()) * w["canvas_len"]
    bytes_tk = kept_rows * V * 4
    peak, peak_kind = _peak_hbm()
    achieved = bytes_rs / (rs_avg_ms / 1e3) / 1e9
    p2_ms = kernel_ms["split_pass2"]
    p1_ms = kernel_ms["split_pass1"]
    achieved_p2 = bytes_rs / (p2_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved_p2, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved_p2 / peak, 4), "traffic": _traffic_from_profile(WORKLOAD, rows),
                "kernel": "split_pass2 (probabilities, Gumbel race, top-k candidates)",
                "peak_kind": f"{peak_kind} copy bandwidth",
                "bytes_per_launch": bytes_rs, "avg_launch_ms": round(p2_ms, 4),
                "launches_averaged": kernel_calls}

    out = {"metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic (seeded N(0,3^2) + one +8 spike per row, temps U[0.5,1.5])",
           "config": {"workload": WORKLOAD_TEXT[WORKLOAD],
                      "rows": rows, "vocab": V, "row_stride": stride, "k": k,
                      "kept_rows": kept_rows,
                      "l2": f"inputs ({rows * V * 4 / 1e9:.1f} GB) larger than L2 (126 MB); "
                            "no flush"},
           "roofline": roofline,
           "kernels": {"row_stats_topk": {"avg_ms": round(rs_avg_ms, 4),
                                          "rows_per_s": round(rows / (rs_avg_ms / 1e3), 1),
                                          "gbs": round(achieved, 1),
                                          "frac_of_peak": round(achieved / peak, 4),
                                          "note": "the whole call over the algorithmic bytes of "
                                                  "one read and one write"},
                       "per_kernel_ms": {k_: round(v_, 4) for k_, v_ in kernel_ms.items()},
                       "split_pass1": {"avg_ms": round(p1_ms, 4),
                                       "gbs_read": round(rows * V * 4 / (p1_ms / 1e3) / 1e9, 1),
                                       "frac_of_peak": round(rows * V * 4 / (p1_ms / 1e3) / 1e9
                                                             / peak, 4)},
                       "row_stats_alone": {"avg_ms": round(sep_rs_ms, 4),
                                           "gbs": round(bytes_rs / (sep_rs_ms / 1e3) / 1e9, 1),
                                           "frac_of_peak": round(bytes_rs / (sep_rs_ms / 1e3)
                                                                 / 1e9 / peak, 4)},
                       "topk_logprobs": {"avg_ms": round(tk_avg_ms, 4),
                                         "gbs_read": round(bytes_tk / (tk_avg_ms / 1e3) / 1e9, 1),
                                         "frac_of_peak": round(bytes_tk / (tk_avg_ms / 1e3) / 1e9
                                                               / peak, 4)},
                       "stash_converged_logprobs": {
                           "avg_ms": round(stash_avg_ms, 4),
                           "gbs_read": round(bytes_tk / (stash_avg_ms / 1e3) / 1e9, 1),
                           "frac_of_peak": round(bytes_tk / (stash_avg_ms / 1e3) / 1e9 / peak, 4),
                           "note": "the kept rows' stash (argmax + top-k) over its algorithmic bytes, one "
                                   "read per kept row (the two passes read it twice)"}},
           # per step: list of rows, pass 1, merge, pass 2, finish, exact top-k
           "gpu_launches": 6 * args.steps,
           "clocks": clocks}

    # end to end through the public API from pinned host memory
    if not args.no_e2e:
        out["e2e"] = _e2e(args, drs, w, rank, world, row0, temps_all, keep_all, k)
    if rows != workloads.WORKLOADS[WORKLOAD].rows:
        out["config"]["workload"] = (f"{WORKLOAD} recipe at {rows} x {V} (a smaller case, "
                                     "not the headline workload)")
        out["config"]["l2"] = "no flush"
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        out["cpu_baseline"] = _cpu_baseline(logits, w, seconds=args.cpu_seconds)
    del logits, probs
    return out


def kernel_source_hash():
    """sha256 over the sources of the row kernels: a traffic figure taken
    from an ncu capture is used only while they are unchanged."""
    import hashlib
    h = hashlib.sha256()
    for rel in ("vocab_row_sampling_gb300/csrc/row_split.cu",
                "vocab_row_sampling_gb300/csrc/drs_device.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic_from_profile(workload, rows):
    """DRAM bytes (read + write) per launch of pass 2, from the committed
    ncu capture, if it was taken on the current kernel sources and covers
    this workload at this number of rows (else null)."""
    path = os.path.join(ROOT, "profiles", "split_pass2_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_sha256") != kernel_source_hash():
            return None
        if d.get("workload_key") != workload or d.get("rows") != rows:
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


def _e2e(args, drs, w, rank, world, row0, temps_all, keep, k):
    rows, V = w["rows"], w["vocab"]
    host = torch.empty(rows, V, dtype=torch.float32, pin_memory=True)
    host.copy_(w["logits"][:, :V].cpu())
    dev = torch.device("cuda")
    d_logits = torch.empty(rows, V, dtype=torch.float32, device=dev)
    temps_h = temps_all.cpu().pin_memory()
    keep_h = keep.cpu().pin_memory()
    d_temps = torch.empty_like(temps_all)
    d_keep = torch.empty_like(keep)
    outs_h = {"argmax": torch.empty(rows, dtype=torch.int64, pin_memory=True),
              "sample": torch.empty(rows, dtype=torch.int64, pin_memory=True),
              "entropy": torch.empty(rows, dtype=torch.float32, pin_memory=True),
              "ids": torch.empty(rows, k, dtype=torch.int32, pin_memory=True),
              "lps": torch.empty(rows, k, dtype=torch.float32, pin_memory=True)}
    argmax = torch.empty(rows, dtype=torch.int64, device=dev)
    sample = torch.empty(rows, dtype=torch.int64, device=dev)
    entropy = torch.empty(rows, dtype=torch.float32, device=dev)
    probs = torch.empty(rows, V, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(rows, k, dtype=torch.int32, device=dev)
    lps = torch.empty(rows, k, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    h2d = host.numel() * 4 + temps_h.numel() * 4 + keep_h.numel()
    d2h = rows * (8 + 8 + 4) + rows * k * (4 + 4)

    # The host-to-device copy (about 211 GB/s on this machine, whichever way
    # it is issued) dominates: the rows go over in chunks on a copy stream,
    # each chunk's call starting once its rows have landed (row0 keeps the
    # results those of one call), so the copy of chunk c + 1 overlaps the
    # compute of chunk c. A chunk's copy in the next step waits for its
    # compute in this one.
    nchunk = 8 if rows % (8 * w["canvas_len"]) == 0 else 1
    ch = rows // nchunk
    copy_stream = torch.cuda.Stream()
    landed = [torch.cuda.Event() for _ in range(nchunk)]
    done = [torch.cuda.Event() for _ in range(nchunk)]
    ws = drs.workspace(drs.drs_row_stats_topk_workspace_bytes(ch, V, k), dev)
    for e in done:
        e.record(stream)

    def step():
        d_temps.copy_(temps_h, non_blocking=True)
        d_keep.copy_(keep_h, non_blocking=True)
        for c in range(nchunk):
            r0, r1 = c * ch, (c + 1) * ch
            copy_stream.wait_event(done[c])
            with torch.cuda.stream(copy_stream):
                d_logits[r0:r1].copy_(host[r0:r1], non_blocking=True)
                landed[c].record(copy_stream)
            stream.wait_event(landed[c])
            drs.drs_row_stats_topk(d_logits[r0:r1], d_temps, w["canvas_len"], 0, argmax[r0:r1],
                                   sample[r0:r1], entropy[r0:r1], drs.DRS_PROBS_BF16,
                                   probs[r0:r1], d_keep, k, ids[r0:r1], lps[r0:r1], ws, stream,
                                   row0=row0 + r0)
            done[c].record(stream)
        outs_h["argmax"].copy_(argmax, non_blocking=True)
        outs_h["sample"].copy_(sample, non_blocking=True)
        outs_h["entropy"].copy_(entropy, non_blocking=True)
        outs_h["ids"].copy_(ids, non_blocking=True)
        outs_h["lps"].copy_(lps, non_blocking=True)

    steps = max(2, min(args.steps, 10))
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    _barrier(world)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    ms = _max_over_ranks(start.elapsed_time(stop), world)
    del host, d_logits, probs
    return {"value": round(world * rows * steps / (ms / 1e3), 1), "unit": "rows/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / steps, 3), "steps": steps,
            "pipeline": f"{nchunk} row chunks, copy of chunk c+1 overlapping compute of chunk c"}


def _cpu_baseline(logits_dev, w, seconds=15.0, threads=None):
    """The oracle, as it stands, on rows of the same batch until about
    `seconds` of wall time; rows/s over the host threads it used."""
    import oracle
    threads = threads or (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                          else os.cpu_count())
    oracle.build()
    rows = w["rows"]
    cl = w["canvas_len"]
    temps = w["temps"].cpu().numpy()
    keep = w["keep"].cpu().numpy()
    done = 0
    t0 = time.perf_counter()
    batch = threads
    while time.perf_counter() - t0 < seconds and done < rows:
        sel = np.arange(done, min(rows, done + batch))
        x = np.ascontiguousarray(logits_dev[torch.as_tensor(sel, device=logits_dev.device)]
                                 .cpu().numpy())
        tr = temps[sel // cl]
        oracle.row_stats_rows(x, sel, tr, 0, oracle.PROBS_BF16, threads=threads)
        kept = sel[keep[sel // cl] != 0]
        if kept.size:
            xk = np.ascontiguousarray(x[np.isin(sel, kept)])
            oracle.topk_rows(xk, temps[kept // cl], w["k"], threads=threads)
        done += sel.size
    el = time.perf_counter() - t0
    return {"value": round(done / el, 2), "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"first {done} rows of the {WORKLOAD} batch (row stats + top-k of kept rows), "
                      f"{el:.1f} s wall"}


# ---------------------------------------------------------- reference arm

def _run_reference(args, world, rank):
    """The CPU oracle timed on the host cores: each step a bounded sample of
    the step workload (rows generated with the same recipe on the CPU)."""
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample_rows = max(threads, 2 * threads)
    w = workloads.make(WORKLOAD, device="cpu", rows=sample_rows)
    V = w["vocab"]
    x = np.ascontiguousarray(w["logits"][:, :V].numpy())
    temps = w["temps"].numpy()
    keep = w["keep"].numpy()
    cl = w["canvas_len"]
    sel = np.arange(sample_rows)

    def step():
        oracle.row_stats_rows(x, sel, temps[sel // cl], 0, oracle.PROBS_BF16, threads=threads)
        kept = sel[keep[sel // cl] != 0]
        if kept.size:
            oracle.topk_rows(np.ascontiguousarray(x[kept]), temps[kept // cl], w["k"],
                             threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = sample_rows * args.steps / el
    sample = (f"{sample_rows} rows of the step workload per step (row stats with bf16 probs "
              f"+ top-k 20 of kept rows), CPU-generated with the same recipe")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "step: 2048 x 262144 fp32 logits (bounded row sample on the "
                                   "host), bf16 probs, top-k 20 on the converged slots",
                       "rows_per_step": sample_rows, "vocab": V},
            "cpu_baseline": {"value": round(value, 3), "unit": "rows/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--rows", type=int, default=None,
                    help="rows per GPU (multiple of the canvas length); default: the full batch")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--workload", default="step", choices=sorted(WORKLOAD_TEXT),
                    help="step (the headline) or wide (rows of 2^21 columns)")
    args = ap.parse_args()
    global WORKLOAD
    WORKLOAD = args.workload
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank == 0:
            print(json.dumps(_run_reference(args, world, rank)), flush=True)
        return
    world, rank, local = _dist()
    out = _run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
