"""Benchmark of the DiffusionGemma row-statistics hot path on GB300.

One step = one pass of the whole path over one batch of the headline
workload ("step" unless --workload says otherwise): drs_row_stats_topk,
the row statistics (argmax, Gumbel-max sample, entropy, bf16 softmax) of
2048 x 262144 fp32 logits and the top-k logprobs (k = 20) of the rows of the
converged (even) slots. Inputs are synthetic (workloads.py) and resident in
HBM when the timed region starts; at 2.1 GB they are larger than L2, so no
flush is needed between steps.

Prints ONE JSON line (rank 0). `value` is rows/s over all GPUs. `roofline`
describes the whole call, which is what the metric names: its algorithmic
bytes (every logit read once, every probability written once: rows*V*4 +
rows*V*2) over the call's average CUDA-event time; its `dominant_kernel`
entry gives the same for the cluster kernel alone (the rows it takes, over
its own time from the library's per-kernel events, recorded during a second
run of the timed steps: the events cost about 15 us per call, so the steps
whose time gives `value` run without them). `kernels` gives every kernel of
the call, the call with the two streaming passes alone, and the separate
calls (drs_row_stats, drs_topk_logprobs, the stash) timed briefly.
`workloads` times the other four workloads of the task the same way
(rows/s, GB/s and fraction of peak, with the oracle's rows/s on the host
beside each and a parity check on sampled rows). `e2e` repeats the step
through the public API from pinned host buffers, copies included;
`cpu_baseline` times the CPU oracle on rows of the same batch, and `parity`
compares those rows with the GPU's results of the last timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --rows 256 --no-e2e --cpu-seconds 0 --no-workloads
      (a smaller case of the same workload, e.g. for a counter capture; not
      a headline number)
  python bench.py --workload strided --rows 256 --no-e2e --cpu-seconds 0 --no-workloads
      (the eight-seed call of the strided workload as the step)
Under torchrun each rank runs its own batch (weak scaling, rows keyed by
global row index so results equal one big batch); no collective touches
the data path.
"""
from __future__ import annotations

import argparse
import json
import math
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
    "large": "large: 8192 x 262144 fp32 logits (peaked rows), fp16 probs, top-k 20, all kept; "
             "not the headline workload",
    "strided": "strided: 2048 x 262144 fp32 logits in rows of stride 262208 (NaN pad), no probs, "
               "8 noise seeds in one call; not the headline workload",
    "adversarial": "adversarial: 1024 x 131072 fp32 (-inf, constant and one-hot rows), bf16 probs, "
                   "top-k 64 on Bernoulli(1/2) slots; not the headline workload",
    "tiny": "tiny: 64 x 8192 fp32 (ties), bf16 probs, top-k 8; not the headline workload",
}
OTHER_WORKLOADS = ("large", "strided", "adversarial", "tiny")
FALLBACK_HBM_GBS = 6800.0
NEAR_TIE_REL = 1e-5  # the sample tolerance of the method: near ties are counted
TRAFFIC_PROFILE = os.path.join("profiles", "row_stats_call_traffic.json")


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


class StepOutputs:
    """Output tensors of one call of a workload (top-k rows of unconverged
    slots keep the -1 / NaN they were filled with)."""

    def __init__(self, w, dev):
        rows, V, k = w["rows"], w["vocab"], w["k"]
        n_seeds = len(w["seeds"]) if w["name"] == "strided" else 1
        self.argmax = torch.empty(rows, dtype=torch.int64, device=dev)
        self.sample = torch.empty(n_seeds, rows, dtype=torch.int64, device=dev)
        self.entropy = torch.empty(rows, dtype=torch.float32, device=dev)
        pdt = {1: torch.bfloat16, 2: torch.float16}.get(w["probs_dtype"])
        self.probs = None if pdt is None else torch.empty(rows, V, dtype=pdt, device=dev)
        self.ids = torch.full((rows, max(k, 1)), -1, dtype=torch.int32, device=dev)
        self.lps = torch.full((rows, max(k, 1)), float("nan"), dtype=torch.float32, device=dev)


def _call_fn(drs, w, logits, temps_all, keep_all, out, stream, row0=0):
    """The workload's call: drs_row_stats_seeds for the multi-seed strided
    workload, drs_row_stats_topk (top-k of the converged rows) otherwise."""
    rows, V, k, cl = w["rows"], w["vocab"], w["k"], w["canvas_len"]
    dev = logits.device
    if w["name"] == "strided":
        ws = drs.workspace(drs.drs_row_stats_seeds_workspace_bytes(rows, V, len(w["seeds"])), dev)
        return lambda: drs.drs_row_stats_seeds(logits, temps_all, cl, w["seeds"], out.argmax,
                                               out.sample, out.entropy, w["probs_dtype"],
                                               out.probs, ws, stream, row0=row0)
    ws = drs.workspace(drs.drs_row_stats_topk_workspace_bytes(rows, V, k), dev)
    return lambda: drs.drs_row_stats_topk(logits, temps_all, cl, 0, out.argmax, out.sample[0],
                                          out.entropy, w["probs_dtype"], out.probs, keep_all, k,
                                          out.ids, out.lps, ws, stream, row0=row0)


def _algorithmic_bytes(w):
    """One read of every logit and one write of every probability (the pad
    columns of a strided buffer are never read)."""
    pb = 2 if w["probs_dtype"] else 0
    return w["rows"] * w["vocab"] * (4 + pb)


def _time_calls(call, stream, n, warmup=2):
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    evs[0].record(stream)
    for _ in range(n):
        call()
    evs[1].record(stream)
    torch.cuda.synchronize()
    return evs[0].elapsed_time(evs[1]) / n


def _run_ours(args, world, rank, local):
    import vocab_row_sampling_gb300 as drs
    drs.load(build_if_missing=True)
    torch.cuda.set_device(local)
    if args.two_pass:
        drs.drs_test_two_pass(True)
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
    out = StepOutputs(w, dev)
    call = _call_fn(drs, w, logits, temps_all, keep_all, out, stream, row0)

    def step():
        call()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if drs.drs_get_device_error() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    def timed():
        # the steps back to back: events only around all of them (an event
        # between two calls holds the next one back)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            # the warm-up steps again once the sampler runs: its start-up
            # pause leaves the GPU idle, and a GPU that has idled (even for
            # the synchronize below) runs its next milliseconds of work about
            # 20% slower, which the default 100 steps amortise
            for _ in range(args.warmup):
                step()
            torch.cuda.synchronize()
            _barrier(world)
            torch.cuda.synchronize()
            start.record(stream)
            for _ in range(args.steps):
                step()
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
        return total_ms, clk.summary(), drs.drs_kernel_times()

    total_ms, clocks, ktimes = timed()
    if _clocks_rejected(clocks):
        total_ms, clocks, ktimes = timed()
        clocks["remeasured"] = True
    kernel_ms, kernel_calls = ktimes
    if drs.drs_get_device_error() != 0:
        raise RuntimeError("device-side wait timed out during the timed region")
    call_ms = total_ms / args.steps  # this rank's call, back to back
    total_ms = _max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = world * rows * args.steps / (total_ms / 1e3)

    peak, peak_kind = _peak_hbm()
    bytes_call = _algorithmic_bytes(w)
    achieved = bytes_call / (call_ms / 1e3) / 1e9
    # the dominant kernel: the cluster kernel on the rows it takes (all of
    # them, or the head of the list when the two passes take the tail on
    # the SMs its clusters leave), else pass 2 of the two passes
    plan = drs.cluster_rows(rows, V, k if w["name"] != "strided" else 0,
                            len(w["seeds"]) if w["name"] == "strided" else 1, w["probs_dtype"])
    if plan is not None and kernel_ms.get("split_cluster", 0.0) > 0.01:
        dk_name, dk_ms, dk_rows = "split_cluster", kernel_ms["split_cluster"], plan["head"]
    else:
        dk_name, dk_ms, dk_rows = "split_pass2", kernel_ms["split_pass2"], rows
    dk_bytes = dk_rows * V * (4 + (2 if w["probs_dtype"] else 0))
    dk_gbs = dk_bytes / (dk_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": _traffic_from_profile(WORKLOAD, rows),
                "kernel": "drs_row_stats_topk, the whole call" if w["name"] != "strided"
                          else "drs_row_stats_seeds, the whole call",
                "peak_kind": f"{peak_kind} copy bandwidth",
                "bytes_per_launch": bytes_call, "avg_launch_ms": round(call_ms, 4),
                "traffic_scope": "dram__bytes_read.sum + dram__bytes_write.sum summed over the "
                                 "kernels of one call (ncu capture, profiles/)",
                "dominant_kernel": {"name": dk_name, "rows": dk_rows, "avg_ms": round(dk_ms, 4),
                                    "bytes_per_launch": dk_bytes, "achieved": round(dk_gbs, 1),
                                    "frac": round(dk_gbs / peak, 4),
                                    "launches_averaged": kernel_calls}}
    if plan is not None:
        roofline["split"] = {"cluster_rows": plan["head"], "two_pass_rows": plan["tail"],
                             "cluster_size": plan["cluster_size"],
                             "clusters_resident": plan["clusters"],
                             "free_sms_for_the_two_passes": plan["free_sms"]}

    kernels = {"call": {"avg_ms": round(call_ms, 4), "rows_per_s": round(rows / (call_ms / 1e3), 1),
                        "gbs": round(achieved, 1), "frac_of_peak": round(achieved / peak, 4)},
               "per_kernel_ms": {k_: round(v_, 4) for k_, v_ in kernel_ms.items()},
               "per_kernel_note": "events on the caller's stream; with the two passes beside the "
                                  "cluster kernel their kernels run on a second stream and are "
                                  "not in this list"}
    # the same call with the two streaming passes alone (the previous design)
    drs.drs_test_two_pass(True)
    try:
        tp_ms = _time_calls(call, stream, max(3, min(args.steps, 30)))
    finally:
        drs.drs_test_two_pass(args.two_pass)
    kernels["two_passes_alone"] = {"avg_ms": round(tp_ms, 4),
                                   "frac_of_peak": round(bytes_call / (tp_ms / 1e3) / 1e9 / peak, 4)}
    if w["name"] == "step":
        kernels.update(_separate_calls(drs, w, logits, temps, temps_all, keep, out, stream, row0,
                                       peak))
    final = {k_: (None if v_ is None else v_.clone()) for k_, v_ in
             (("argmax", out.argmax), ("sample", out.sample), ("entropy", out.entropy),
              ("probs", out.probs), ("ids", out.ids), ("lps", out.lps))}

    res = {"metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic (workloads.py recipe of the named workload, seeded)",
           "config": {"workload": WORKLOAD_TEXT[WORKLOAD],
                      "rows": rows, "vocab": V, "row_stride": stride, "k": k,
                      "l2": f"inputs ({rows * V * 4 / 1e9:.2f} GB) larger than L2 (126 MB); "
                            "no flush" if rows * V * 4 > 126e6 else "inputs fit L2; no flush"},
           "roofline": roofline,
           "kernels": kernels,
           # per step: the list of rows, the cluster kernel (and the three
           # kernels of the two passes on the second stream), the finish, the
           # exact top-k kernel
           "gpu_launches": _launches_per_call(plan, k) * args.steps,
           "clocks": clocks}

    if not args.no_e2e and w["name"] != "strided":
        res["e2e"] = _e2e(args, drs, w, rank, world, row0, temps_all, keep_all, k)
    if rows != workloads.WORKLOADS[WORKLOAD].rows:
        res["config"]["workload"] = (f"{WORKLOAD} recipe at {rows} x {V} (a smaller case, "
                                     "not the headline workload)")
        res["config"]["l2"] = "no flush"
    if args.two_pass:
        res["config"]["two_pass_only"] = ("every call took the two streaming passes (for profiling them; "
                                          "not the headline configuration)")
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        base, parity = _cpu_baseline(logits, w, final, seconds=args.cpu_seconds)
        res["cpu_baseline"] = base
        res["parity"] = parity
    del final, out, logits
    if rank == 0 and world == 1 and not args.no_workloads and args.rows is None:
        res["workloads"] = {name: _workload_case(drs, name, args, peak)
                            for name in OTHER_WORKLOADS if name != WORKLOAD}
    return res


def _launches_per_call(plan, k):
    if plan is None:
        return 6  # list, pass 1, merge, pass 2, finish, exact top-k
    n = 3 + (3 if plan["tail"] > 0 else 0)  # list, cluster, finish (+ pass 1, merge, pass 2)
    return n + (1 if k > 0 else 0)


def _separate_calls(drs, w, logits, temps, temps_all, keep, out, stream, row0, peak, n=30):
    """drs_row_stats, drs_topk_logprobs and the stash of the converged
    requests, each timed briefly (context for the fused call)."""
    rows, V, k, cl = w["rows"], w["vocab"], w["k"], w["canvas_len"]
    dev = logits.device
    ws_rs = drs.workspace(drs.drs_row_stats_workspace_bytes(rows, V), dev)
    ws_tk = drs.workspace(drs.drs_topk_workspace_bytes(rows, V, k), dev)
    rs_ms = _time_calls(lambda: drs.drs_row_stats(logits, temps_all, cl, 0, out.argmax, out.sample[0],
                                                  out.entropy, drs.DRS_PROBS_BF16, out.probs, ws_rs,
                                                  stream, row0=row0), stream, n)
    tk_ms = _time_calls(lambda: drs.drs_topk_logprobs(logits, temps, cl, keep, k, out.ids, out.lps,
                                                      ws_tk, stream), stream, n)
    n_slots = rows // cl
    req = torch.arange(n_slots, dtype=torch.int32, device=dev)
    valid_all = torch.full((n_slots,), cl, dtype=torch.int32, device=dev)
    st_ids = torch.empty(n_slots, cl, k + 1, dtype=torch.int32, device=dev)
    st_vals = torch.empty(n_slots, cl, k + 1, dtype=torch.float32, device=dev)
    st_ranks = torch.empty(n_slots, cl, dtype=torch.int32, device=dev)
    ws_st = drs.workspace(drs.drs_stash_workspace_bytes(n_slots, cl, V, k), dev)
    st_ms = _time_calls(lambda: drs.drs_stash_converged_logprobs(
        logits, cl, req, req, keep, valid_all, temps, k, None, None, st_ids, st_vals, st_ranks,
        False, ws_st, stream), stream, n)
    bytes_rs = rows * V * 6
    kept_rows = int(keep[:n_slots].sum().item()) * cl
    bytes_tk = kept_rows * V * 4
    return {"row_stats_alone": {"avg_ms": round(rs_ms, 4),
                                "frac_of_peak": round(bytes_rs / (rs_ms / 1e3) / 1e9 / peak, 4)},
            "topk_logprobs": {"avg_ms": round(tk_ms, 4), "kept_rows": kept_rows,
                              "frac_of_peak": round(bytes_tk / (tk_ms / 1e3) / 1e9 / peak, 4),
                              "note": "over kept_rows*V*4 bytes: one read of each kept row"},
            "stash_converged_logprobs": {"avg_ms": round(st_ms, 4),
                                         "frac_of_peak": round(bytes_tk / (st_ms / 1e3) / 1e9 / peak, 4),
                                         "note": "the kept rows' stash (argmax + top-k), over one "
                                                 "read of each kept row"}}


def _workload_case(drs, name, args, peak, sample_rows=6, steps=20):
    """One of the task's other workloads: its call timed, rows/s, GB/s and
    fraction of peak over one read and one write; the oracle's rows/s on a
    few of its rows on the host; those rows compared with the GPU's."""
    import oracle
    w = workloads.make(name, device="cuda")
    rows, V, cl = w["rows"], w["vocab"], w["canvas_len"]
    logits = w["logits"][:, :V]
    temps, keep = w["temps"].cuda(), w["keep"].cuda()
    out = StepOutputs(w, logits.device)
    stream = torch.cuda.current_stream()
    call = _call_fn(drs, w, logits, temps, keep, out, stream)
    ms = _time_calls(call, stream, steps)
    if drs.drs_get_device_error() != 0:
        raise RuntimeError(f"device-side wait timed out in workload {name}")
    nb = _algorithmic_bytes(w)
    gbs = nb / (ms / 1e3) / 1e9
    sel = np.unique(np.linspace(0, rows - 1, min(sample_rows, rows)).astype(np.int64))
    if rows <= 64:
        sel = np.arange(rows)
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    oracle.build()
    x = np.ascontiguousarray(logits[torch.as_tensor(sel, device=logits.device)].cpu().numpy())
    tr = w["temps"].cpu().numpy()[sel // cl]
    seeds = w["seeds"] if name == "strided" else [0]
    t0 = time.perf_counter()
    refs = [oracle.row_stats_rows(x, sel, tr, sd, w["probs_dtype"], threads=threads) for sd in seeds]
    kept = sel[w["keep"].cpu().numpy()[sel // cl] != 0] if w["k"] else sel[:0]
    topk_ref = None
    if kept.size:
        topk_ref = oracle.topk_rows(np.ascontiguousarray(x[np.isin(sel, kept)]),
                                    w["temps"].cpu().numpy()[kept // cl], w["k"], threads=threads)
    el = time.perf_counter() - t0
    gpu = {"argmax": out.argmax.cpu().numpy()[sel], "entropy": out.entropy.cpu().numpy()[sel],
           "sample": out.sample.cpu().numpy()[:, sel],
           "probs": None if out.probs is None else
           out.probs[torch.as_tensor(sel, device=logits.device)].view(torch.int16).cpu().numpy().view(np.uint16),
           "ids": out.ids.cpu().numpy()[kept], "lps": out.lps.cpu().numpy()[kept]}
    par = _compare(gpu, refs, topk_ref, w["probs_dtype"])
    res = {"rows": rows, "vocab": V, "row_stride": w["row_stride"], "k": w["k"],
           "avg_ms": round(ms, 4), "rows_per_s": round(rows / (ms / 1e3), 1),
           "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
           "bytes_per_call": nb,
           "oracle_rows_per_s": round(len(sel) * len(seeds) / el, 2), "oracle_threads": threads,
           "parity_sampled_rows": par}
    if name == "strided":
        res["note"] = f"drs_row_stats_seeds with {len(seeds)} seeds (one read, a sample per seed)"
    del w, logits, out
    torch.cuda.empty_cache()
    return res


def _compare(gpu, refs, topk_ref, probs_dtype):
    """Counts and worst errors of the GPU's rows against the oracle's (the
    tolerances of the method: argmax and top-k ids exact; samples exact
    except near ties, counted; entropy and logprobs within 1e-4; probs within
    one code)."""
    res = {"rows": int(gpu["argmax"].size),
           "argmax_mismatch": int(np.sum(gpu["argmax"] != refs[0]["argmax"]))}
    hard = near = 0
    for i, ref in enumerate(refs):
        diff = np.flatnonzero(gpu["sample"][i] != ref["sample"])
        tie = ref["sample_gap"][diff] <= NEAR_TIE_REL * np.maximum(1.0, np.abs(ref["sample_best"][diff]))
        near += int(tie.sum())
        hard += int((~tie).sum())
    res["sample_mismatch_outside_near_ties"] = hard
    res["sample_near_ties"] = near
    res["entropy_max_abs_err"] = float(np.max(np.abs(gpu["entropy"].astype(np.float64) - refs[0]["entropy"])))
    if probs_dtype and gpu["probs"] is not None:
        d = np.abs(gpu["probs"].astype(np.int64) - refs[0]["probs"].astype(np.int64))
        res["probs_max_code_diff"] = int(d.max()) if d.size else 0
    if topk_ref is not None:
        ri, rl = topk_ref
        res["topk_rows"] = int(ri.shape[0])
        res["topk_id_mismatch_rows"] = int(np.sum(np.any(gpu["ids"] != ri, axis=1)))
        both = np.isfinite(rl) & np.isfinite(gpu["lps"])
        err = np.abs(gpu["lps"].astype(np.float64) - rl)[both]
        rel = err / np.maximum(1e-4, np.spacing(np.abs(rl[both]).astype(np.float32)).astype(np.float64))
        res["logprob_max_abs_err"] = float(err.max()) if err.size else 0.0
        res["logprob_within_tolerance"] = bool(np.all(rel <= 1.0)) if err.size else True
    return res


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


def kernel_source_hash():
    """sha256 over the code of the row kernels' sources (comments and blank
    lines dropped): a traffic figure taken from an ncu capture is used only
    while that code is unchanged."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in ("vocab_row_sampling_gb300/csrc/row_split.cu",
                "vocab_row_sampling_gb300/csrc/row_cluster.cu",
                "vocab_row_sampling_gb300/csrc/row_common.cuh",
                "vocab_row_sampling_gb300/csrc/drs_device.cuh"):
        with open(os.path.join(ROOT, rel)) as f:
            code = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        for line in code.splitlines():
            line = line.split("//", 1)[0].rstrip()
            if line.strip():
                h.update(line.encode() + b"\n")
    return h.hexdigest()


def _traffic_from_profile(workload, rows):
    """DRAM bytes (read + write) of one call, summed over its kernels, from
    the committed ncu capture, if it was taken on the current kernel sources
    and covers this workload at this number of rows (else null)."""
    path = os.path.join(ROOT, TRAFFIC_PROFILE)
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_sha256") != kernel_source_hash():
            return None
        if d.get("workload_key") != workload or d.get("rows") != rows:
            return None
        return d.get("dram_bytes_per_call")
    except Exception:
        return None


def _cpu_baseline(logits_dev, w, final, seconds=15.0, threads=None):
    """The oracle, as it stands, on rows of the same batch until about
    `seconds` of oracle time (row statistics, with the top-k of the kept
    rows); rows/s over the host threads it used. Those rows are also compared
    with the GPU's results of the last timed step (the parity block)."""
    import oracle
    threads = threads or (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                          else os.cpu_count())
    oracle.build()
    rows = w["rows"]
    cl = w["canvas_len"]
    temps = w["temps"].cpu().numpy()
    keep = w["keep"].cpu().numpy()
    seeds = w["seeds"] if w["name"] == "strided" else [0]
    g_argmax = final["argmax"].cpu().numpy()
    g_sample = final["sample"].cpu().numpy()
    g_entropy = final["entropy"].cpu().numpy()
    g_ids = final["ids"].cpu().numpy()
    g_lps = final["lps"].cpu().numpy()
    agg = {"rows": 0, "argmax_mismatch": 0, "sample_mismatch_outside_near_ties": 0,
           "sample_near_ties": 0, "entropy_max_abs_err": 0.0}
    if w["probs_dtype"]:
        agg["probs_max_code_diff"] = 0
    if w["k"]:
        agg.update({"topk_rows": 0, "topk_id_mismatch_rows": 0, "logprob_max_abs_err": 0.0,
                    "logprob_within_tolerance": True})
    done = 0
    el = 0.0
    batch = threads
    while el < seconds and done < rows:
        sel = np.arange(done, min(rows, done + batch))
        sel_dev = torch.as_tensor(sel, device=logits_dev.device)
        x = np.ascontiguousarray(logits_dev[sel_dev].cpu().numpy())
        tr = temps[sel // cl]
        kept = sel[keep[sel // cl] != 0] if w["k"] else sel[:0]
        t0 = time.perf_counter()
        refs = [oracle.row_stats_rows(x, sel, tr, sd, w["probs_dtype"], threads=threads) for sd in seeds]
        topk_ref = None
        if kept.size:
            topk_ref = oracle.topk_rows(np.ascontiguousarray(x[np.isin(sel, kept)]), temps[kept // cl],
                                        w["k"], threads=threads)
        el += time.perf_counter() - t0
        gpu = {"argmax": g_argmax[sel], "sample": g_sample[:, sel], "entropy": g_entropy[sel],
               "probs": None if final["probs"] is None else
               final["probs"][sel_dev].view(torch.int16).cpu().numpy().view(np.uint16),
               "ids": g_ids[kept], "lps": g_lps[kept]}
        c = _compare(gpu, refs, topk_ref, w["probs_dtype"])
        for key_ in ("rows", "argmax_mismatch", "sample_mismatch_outside_near_ties", "sample_near_ties",
                     "topk_rows", "topk_id_mismatch_rows"):
            if key_ in c:
                agg[key_] += c[key_]
        for key_ in ("entropy_max_abs_err", "probs_max_code_diff", "logprob_max_abs_err"):
            if key_ in c:
                agg[key_] = max(agg[key_], c[key_])
        if "logprob_within_tolerance" in c:
            agg["logprob_within_tolerance"] &= c["logprob_within_tolerance"]
        done += sel.size
    agg["bar"] = ("argmax and top-k ids exact; samples exact except near ties (the two best "
                  "oracle scores within 1e-5 relative), counted; entropy and logprobs within 1e-4 "
                  "(or one fp32 ulp); probs within one code")
    agg["of_rows"] = rows
    base = {"value": round(done / el, 2), "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"first {done} rows of the {w['name']} batch (row stats"
                      + (" + top-k of kept rows" if w["k"] else "") + f"), {el:.1f} s of oracle time"}
    return base, agg


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
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--rows", type=int, default=None,
                    help="rows per GPU (multiple of the canvas length); default: the full batch")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--workload", default="step", choices=sorted(WORKLOAD_TEXT),
                    help="the workload of a step: step (the headline), or another for a "
                         "separate measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the timings of the other workloads")
    ap.add_argument("--two-pass", action="store_true",
                    help="every call takes the two streaming passes, not the cluster kernel (to "
                         "profile the passes alone; not the headline configuration)")
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
