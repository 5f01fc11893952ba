"""The multi-GPU layout on the CPU: two gloo ranks each own a batch of rows
keyed by global row index (row0 = rank * rows). Together they must give
what one process gives on the concatenated batch. Also checks the bench's
max-over-ranks timing reduction. No GPU; the per-rank compute is the oracle
(the GPU path takes the same row0 and is checked against it in the GPU
parity tests)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, rows, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import workloads
    w = workloads.make("tiny", data_seed=rank, rows=rows)
    cl = w["canvas_len"]
    row0, slot0 = bench.shard_layout(rank, rows, cl)
    temps_all = bench.global_temps(w["temps"], rank, rows, cl).numpy()
    gids = np.arange(row0, row0 + rows)
    x = w["logits"].numpy()
    r = oracle.row_stats_rows(x, gids, temps_all[gids // cl], seed=5,
                              probs_dtype=oracle.PROBS_BF16, threads=2)
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), x=x, temps=w["temps"].numpy(),
             argmax=r["argmax"], sample=r["sample"], entropy=r["entropy"], probs=r["probs"])
    t = bench._max_over_ranks(float(rank + 1) * 1.5, world)
    assert t == 1.5 * world
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_row_sharding_matches_one_process(world, tmp_path):
    rows = 32
    mp.start_processes(_rank_main, args=(world, _free_port(), rows, str(tmp_path)),
                       nprocs=world, start_method="spawn")
    import oracle
    parts = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    x = np.concatenate([p["x"] for p in parts])
    cl = 16
    temps = np.concatenate([p["temps"][: rows // cl] for p in parts])
    ref = oracle.row_stats(x, temps, cl, seed=5, probs_dtype=oracle.PROBS_BF16, threads=4)
    for key in ("argmax", "sample", "entropy", "probs"):
        got = np.concatenate([p[key] for p in parts])
        assert np.array_equal(got, ref[key]), key
