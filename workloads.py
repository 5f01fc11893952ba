"""Seeded synthetic inputs for the DiffusionGemma row-statistics workloads.

This module only draws inputs: it holds none of the sampler's arithmetic and
serves the CUDA path and the CPU oracle alike. Every draw comes from a
``torch.Generator`` seeded with ``data_seed`` on the requested device, so a
workload is reproducible bit for bit on one device type. (CPU and CUDA
generators give different streams; a test that compares the two paths feeds
both the same bytes.)

The workloads (the pages print no benchmark; these stand in for the shapes
the sampler runs on; "wide" exercises rows longer than the configurations'):

  tiny         4 slots x canvas 16 = 64 rows, V = 8192, x ~ N(0, 2^2) with 5%
               of the entries rounded to multiples of 0.25 (ties), temps
               [0, 0.7, 1.0, 1.3], bf16 probs, k = 8, every slot kept.
  step         8 x 256 = 2048 rows, V = 262144, x ~ N(0, 3^2) plus 8.0 at one
               random column per row, temps ~ U[0.5, 1.5], bf16 probs,
               k = 20, even slots kept.
  large        32 x 256 = 8192 rows, V = 262144, peaked rows: background
               N(0, 1) plus 64 random columns per row drawn from N(mu, 1),
               mu ~ U[4, 12] (one mean per component; a column drawn twice
               keeps the larger value), temps ~ U[0.1, 2.0]
               with 8 of the 32 slots exactly 0, fp16 probs, k = 20, all kept.
  strided      2048 rows (8 x 256) of V = 262144 inside a buffer with row
               stride 262208 whose pad columns hold NaN, x ~ N(0, 3^2),
               temps all 1.0, no probs, k = 0, noise seeds 0..7.
  wide         2 x 256 = 512 rows, V = 2097152 (2^21): the step recipe on
               rows eight times longer (slot 0 kept).
  adversarial  8 x 128 = 1024 rows, V = 131072: 10% of rows constant (one
               N(0,1) value), 10% one-hot (0 at one column, -inf elsewhere),
               the rest N(0, 3^2) with 30% of the entries -inf; temps cycle
               {0, 1e-3, 1e-10, 1.0} over slots, bf16 probs, k = 64, keep ~
               Bernoulli(0.5) per slot.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

PROBS_NONE, PROBS_BF16, PROBS_FP16 = 0, 1, 2


@dataclass
class Workload:
    name: str
    slots: int
    canvas_len: int
    vocab: int
    row_stride: int
    probs_dtype: int
    k: int
    seeds: list = field(default_factory=lambda: [0])
    description: str = ""

    @property
    def rows(self) -> int:
        return self.slots * self.canvas_len


WORKLOADS = {
    "tiny": Workload("tiny", 4, 16, 8192, 8192, PROBS_BF16, 8,
                     description="64x8192 fp32, ties, temps [0,0.7,1,1.3], bf16, k=8"),
    "step": Workload("step", 8, 256, 262144, 262144, PROBS_BF16, 20,
                     description="2048x262144 fp32 N(0,9)+spike, bf16, k=20"),
    "large": Workload("large", 32, 256, 262144, 262144, PROBS_FP16, 20,
                      description="8192x262144 fp32 mixture, fp16, k=20"),
    "strided": Workload("strided", 8, 256, 262144, 262208, PROBS_NONE, 0,
                        seeds=list(range(8)),
                        description="2048 rows, stride 262208 NaN pad, no probs, 8 seeds"),
    "wide": Workload("wide", 2, 256, 2097152, 2097152, PROBS_BF16, 20,
                     description="512x2097152 fp32 N(0,9)+spike, bf16, k=20"),
    "adversarial": Workload("adversarial", 8, 128, 131072, 131072, PROBS_BF16, 64,
                            description="1024x131072 fp32 with -inf/constant/one-hot rows, k=64"),
}


def _gen(device, data_seed):
    g = torch.Generator(device=device)
    g.manual_seed(data_seed)
    return g


def make_temps_keep(name: str, data_seed: int = 0):
    """(temps fp32 [slots], keep uint8 [slots]) on the CPU."""
    w = WORKLOADS[name]
    g = _gen("cpu", data_seed + 1000)
    if name == "tiny":
        temps = torch.tensor([0.0, 0.7, 1.0, 1.3], dtype=torch.float32)
        keep = torch.ones(w.slots, dtype=torch.uint8)
    elif name in ("step", "wide"):
        temps = 0.5 + torch.rand(w.slots, generator=g, dtype=torch.float32)
        keep = (torch.arange(w.slots) % 2 == 0).to(torch.uint8)
    elif name == "large":
        temps = 0.1 + 1.9 * torch.rand(w.slots, generator=g, dtype=torch.float32)
        zero = torch.randperm(w.slots, generator=g)[: w.slots // 4]
        temps[zero] = 0.0
        keep = torch.ones(w.slots, dtype=torch.uint8)
    elif name == "strided":
        temps = torch.ones(w.slots, dtype=torch.float32)
        keep = torch.zeros(w.slots, dtype=torch.uint8)
    elif name == "adversarial":
        cyc = torch.tensor([0.0, 1e-3, 1e-10, 1.0], dtype=torch.float32)
        temps = cyc[torch.arange(w.slots) % 4].clone()
        keep = (torch.rand(w.slots, generator=g) < 0.5).to(torch.uint8)
    else:
        raise KeyError(name)
    return temps, keep


def make_logits(name: str, device="cpu", data_seed: int = 0, rows: int | None = None):
    """Logits buffer [rows, row_stride] fp32 on `device`; the first `vocab`
    columns are the logits, pad columns (if any) hold NaN. `rows` (default:
    the workload's) truncates or extends the row count with the same recipe.
    """
    w = WORKLOADS[name]
    R = w.rows if rows is None else rows
    V, stride = w.vocab, w.row_stride
    g = _gen(device, data_seed)
    if name == "tiny":
        x = 2.0 * torch.randn(R, V, generator=g, device=device)
        pick = torch.rand(R, V, generator=g, device=device) < 0.05
        x = torch.where(pick, torch.round(x * 4.0) / 4.0, x)
        buf = x
    elif name in ("step", "strided", "wide"):
        buf = torch.empty(R, stride, device=device, dtype=torch.float32)
        buf[:, :V].normal_(0.0, 3.0, generator=g)
        if stride > V:
            buf[:, V:] = float("nan")
        if name in ("step", "wide"):
            col = torch.randint(0, V, (R,), generator=g, device=device)
            buf[torch.arange(R, device=device), col] += 8.0
    elif name == "large":
        buf = torch.randn(R, V, generator=g, device=device)
        mu = 4.0 + 8.0 * torch.rand(64, generator=g, device=device)
        cols = torch.randint(0, V, (R, 64), generator=g, device=device)
        vals = mu[None, :] + torch.randn(R, 64, generator=g, device=device)
        # columns drawn twice for a row keep the larger value (an order-free
        # rule, so the batch is the same bytes on every run)
        buf.scatter_reduce_(1, cols, vals, reduce="amax", include_self=False)
    elif name == "adversarial":
        buf = 3.0 * torch.randn(R, V, generator=g, device=device)
        masked = torch.rand(R, V, generator=g, device=device) < 0.3
        buf[masked] = float("-inf")
        kind = torch.rand(R, generator=g, device=device)
        const_rows = kind < 0.1
        onehot_rows = (kind >= 0.1) & (kind < 0.2)
        const_val = torch.randn(R, generator=g, device=device)
        hot_col = torch.randint(0, V, (R,), generator=g, device=device)
        cr = const_rows.nonzero().flatten()
        if cr.numel():
            buf[cr] = const_val[cr][:, None].expand(-1, V)
        orow = onehot_rows.nonzero().flatten()
        if orow.numel():
            buf[orow] = float("-inf")
            buf[orow, hot_col[orow]] = 0.0
    else:
        raise KeyError(name)
    return buf.to(torch.float32).contiguous()


def make(name: str, device="cpu", data_seed: int = 0, rows: int | None = None):
    """Everything one workload needs: dict with logits buffer, vocab,
    row_stride, temps, keep, canvas_len, seeds, probs_dtype, k."""
    w = WORKLOADS[name]
    temps, keep = make_temps_keep(name, data_seed)
    R = w.rows if rows is None else rows
    slots_needed = -(-R // w.canvas_len)
    if slots_needed > temps.numel():  # extended row counts reuse the cycle
        reps = -(-slots_needed // temps.numel())
        temps = temps.repeat(reps)[:slots_needed]
        keep = keep.repeat(reps)[:slots_needed]
    return {
        "name": name,
        "logits": make_logits(name, device, data_seed, rows=R),
        "rows": R,
        "vocab": w.vocab,
        "row_stride": w.row_stride,
        "temps": temps.to(device),
        "keep": keep.to(device),
        "canvas_len": w.canvas_len,
        "seeds": list(w.seeds),
        "probs_dtype": w.probs_dtype,
        "k": w.k,
    }
