"""The benchmark's byte accounting (the roofline's algorithmic bytes), on CPU.

The accounting rule: every needed logit row read once (target rows; draft
rows of sampled sequences only, greedy sequences need none), plus one
row-equivalent per sampled sequence for the resample, plus the small
per-row and per-sequence tensors.  The totals are checked against the
sizes of the three bandwidth workloads worked out by hand from their
shapes (B, k, V, dtype, greedy mix), and the draft and verify passes of the
round against their own parts.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads

SMALL_SLACK = 1 << 20  # the small tensors (offsets, uniforms, outputs) stay far below 1 MiB here


def big_part(n_rows, V, s):
    return n_rows * V * s


@pytest.mark.parametrize("cfg,expect_rows", [
    # B=64, k=5, all sampled: 64*6 target rows + 64*5 draft rows + 64 resample row-equivalents
    (3, 64 * 6 + 64 * 5 + 64),
    # B=256, k=8, odd sequences greedy: 256*9 target rows + the 128 sampled sequences' 128*8
    # draft rows + 128 resample row-equivalents
    (4, 256 * 9 + 128 * 8 + 128),
])
def test_verify_bytes_of_the_uniform_workloads(cfg, expect_rows):
    w = workloads.make_config(cfg)
    ab = workloads.algorithmic_bytes(w)
    big = big_part(expect_rows, w.V, 2)
    assert big <= ab["verify"] <= big + SMALL_SLACK
    assert ab["rows_verified"] == w.rows_target + w.rows_draft


def test_verify_bytes_of_the_ragged_workload():
    """B=512, k_b uniform in 1..10, all sampled: the row counts come from the
    seeded k_b; every target and draft row is needed, plus 512 resamples."""
    w = workloads.make_config(5)
    k = np.diff(w.k_offsets)
    assert k.min() >= 1 and k.max() <= 10 and (w.temperature > 0).all()
    R_d = int(k.sum())
    R_t = R_d + w.B
    ab = workloads.algorithmic_bytes(w)
    big = big_part(R_t + R_d + w.B, w.V, 2)
    assert big <= ab["verify"] <= big + SMALL_SLACK
    # the round: the draft pass reads every draft row once; the verify pass
    # then reads the target rows and the resample row-equivalents only
    assert big_part(R_d, w.V, 2) <= ab["draft_sample"] <= big_part(R_d, w.V, 2) + SMALL_SLACK
    assert big_part(R_t + w.B, w.V, 2) <= ab["verify_lse"] <= big_part(R_t + w.B, w.V, 2) + SMALL_SLACK
    # one round (both passes) moves what the verify call's accounting counts: the draft
    # rows once (in the draft pass), the target rows and the resamples once (in the verify
    # pass), within the small tensors
    assert abs((ab["draft_sample"] + ab["verify_lse"]) - ab["verify"]) <= SMALL_SLACK
