"""Writes tests/golden/flag_counts.json: for each of the five workloads (fixed
seeds), how many decisions the fp64 oracle takes within FLAG_MARGIN = 1e-5
of a boundary.

A sequence is flagged when a decision it took has margin <= 1e-5 (a uniform
within 1e-5 of an accept threshold alpha_i, or of the CDF step of the drawn
token); a draft row likewise for its draw.  The flagging rule is the verify
step's parity contract (tokens bit-exact except where a uniform lies within
1e-5 of a decision boundary; such cases are counted and reported).

Only the oracle and the seeded generator run here.  Verify counts use the
oracle's own draft tokens, as the full-size parity tests do.

  python tests/golden/flag_counts.py
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402

FLAG_MARGIN = 1e-5


def counts(w, nthreads):
    ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets, nthreads=nthreads)
    ov = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample, w.temperature,
                       w.k_offsets, nthreads=nthreads)
    return {"sequences": int(w.B), "draft_rows": int(w.rows_draft),
            "verify_flagged": int(((ov.num_accepted >= 0) & (ov.margin <= FLAG_MARGIN)).sum()),
            "draft_flagged": int((ds.margin <= FLAG_MARGIN).sum()),
            "verify_data_errors": int((ov.num_accepted < 0).sum())}


def main():
    out = {"about": "Oracle-flagged decisions (margin <= 1e-5) per workload, written by "
                    "tests/golden/flag_counts.py from the fp64 oracle and the seeded generator.",
           "flag_margin": FLAG_MARGIN, "workloads": {}}
    for cfg in range(1, 6):
        w = workloads.make_config(cfg)
        out["workloads"][w.name] = counts(w, oracle.cores())
        print(w.name, out["workloads"][w.name], flush=True)
    with open(os.path.join(HERE, "flag_counts.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
