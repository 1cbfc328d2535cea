"""The benchmark's reference arm (the fp64 oracle on the host cores) under a
two-rank torchrun on CPU: rank 0 alone prints one JSON line with the
contract's keys, the other rank exits without work, and both exit 0."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "3", "--warmup", "3", "--cpu-seconds", "0.3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "B512_ragged_k1to10_V128256_bf16"
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    assert d["config"] == bench.line_config(workloads.make_config(5), 2)  # the GPU arm's dict, key for key


def test_oracle_parity_counts_flags_and_mismatches():
    """The bench's parity block: outputs equal to the oracle's give no
    mismatch, a flipped token outside the flags is counted."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import oracle
    import workloads
    w = workloads.make_config(2)
    ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
    ov = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample, w.temperature,
                       w.k_offsets)
    p = bench.oracle_parity(w, (ds.tokens.copy(), ov.tokens.copy(), ov.num_accepted.copy()), 2)
    assert p["mismatched_sequences_outside_flags"] == 0 and p["draft_mismatched_rows_outside_flags"] == 0
    assert p["flagged_match"] == p["flagged_sequences"] and p["draft_flagged_match"] == p["draft_flagged_rows"]
    assert p["draft_flagged_rows"] == int((ds.margin <= 1e-5).sum())
    b = int(np.flatnonzero(ov.margin > 1e-5)[0])
    tok = ov.tokens.copy()
    o = int(w.k_offsets[b]) + b
    tok[o] = (tok[o] + 1) % w.V
    p = bench.oracle_parity(w, (ds.tokens.copy(), tok, ov.num_accepted.copy()), 2)
    assert p["mismatched_sequences_outside_flags"] == 1
