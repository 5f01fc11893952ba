"""Write oracle_tiny.json: the oracle's results on small seeded inputs.

These are not values printed by the pages (they print no worked example);
they are a regression fixture of the oracle (oracle/drs_oracle.c), written
by this script, which calls only oracle/ and the seeded input generator.
tests/test_golden.py recomputes them and requires the same results, so a
change to the oracle's arithmetic shows up as a fixture diff.

  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402


ROWS = [0, 17, 33, 40, 49, 63]  # rows of all four slots


def compute():
    w = workloads.make("tiny")
    x = np.ascontiguousarray(w["logits"].numpy())
    temps = w["temps"].numpy()                # [0, 0.7, 1.0, 1.3] over 4 slots of 16 rows
    sel = ROWS
    rows = {"rows": sel}
    r = oracle.row_stats(x, temps, 16, 7, oracle.PROBS_BF16, rows_sel=sel)
    rows["argmax"] = [int(r["argmax"][i]) for i in sel]
    rows["sample"] = [int(r["sample"][i]) for i in sel]
    rows["entropy"] = [float(r["entropy"][i]) for i in sel]
    rows["probs_code_sum"] = [int(r["probs"][i].astype(np.int64).sum()) for i in sel]
    ids, lps = oracle.topk_logprobs(x, temps, 16, np.ones(4, np.uint8), 8, rows_sel=sel)
    topk = {"ids": [ids[i].tolist() for i in sel], "logprobs": [lps[i].tolist() for i in sel]}
    xs = np.array([[1, 3, 3, -np.inf, 0, 2], [0, 0, 0, 0, 0, 0],
                   [5, 4, 3, 2, 1, 0], [-1, -2, -3, -4, -5, -6]], np.float32)
    sid, sval, sr = oracle.stash(xs, 2, [1, 0], [0, 1], [1, 1], [2, 1], [1.0, 0.5], 3, None, None, 2, 5)
    stash = {"ids": sid.tolist(), "values": [[[None if np.isnan(v) else v for v in c] for c in p]
                                             for p in sval.tolist()], "ranks": sr.tolist()}
    return {"note": "oracle results on seeded inputs (see make_golden.py); not values from the pages",
            "row_stats_tiny_seed_7": rows, "topk8_tiny": topk,
            "stash_example": stash}


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
