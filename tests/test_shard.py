"""Sequence sharding of a verify batch over ranks (host logic; CPU, gloo).

The verify step has no cross-sequence data flow, so a batch split into
contiguous sequence ranges and verified rank by rank must give exactly the
full-batch result.  The per-rank compute here is the oracle (the only CPU
implementation); on GPUs each rank calls spec_verify on the same slices.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

from speculative_decoding_verification_61_gb300 import shard


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_ranges_partition_and_balance(world):
    rng = np.random.default_rng(7)
    k = rng.integers(1, 11, size=37)
    ko = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
    rr = shard.shard_ranges(ko, world)
    assert len(rr) == world and rr[0][0] == 0 and rr[-1][1] == 37
    assert all(rr[i][1] == rr[i + 1][0] for i in range(world - 1))
    cost = [int(sum(2 * k[b] + 1 for b in range(b0, b1))) for b0, b1 in rr]
    ideal = sum(2 * k + 1) / world
    # every cut lands within one sequence (at most 21 rows) of the ideal
    assert all(abs(c - ideal) <= world * 21 for c in cost)


def test_more_ranks_than_sequences():
    ko = np.array([0, 3, 5], dtype=np.int32)
    rr = shard.shard_ranges(ko, 5)
    assert rr[0][0] == 0 and rr[-1][1] == 2
    assert sum(b1 - b0 for b0, b1 in rr) == 2
    empty = [s for s in (shard.make_shard(ko, *r) for r in rr) if s.B == 0]
    assert empty and all(s.draft_rows[0] == s.draft_rows[1] for s in empty)


def test_shard_rows_and_rebase():
    ko = np.array([0, 2, 7, 8, 12], dtype=np.int32)
    s = shard.make_shard(ko, 1, 3)
    assert s.draft_rows == (2, 8)
    assert s.target_rows == (3, 11)  # k_offsets[b] + b; k_1 + 1 + k_2 + 1 = 8 rows
    assert s.k_offsets.tolist() == [0, 5, 6]
    with pytest.raises(ValueError):
        shard.make_shard(ko, 3, 2)
    with pytest.raises(ValueError):
        shard.shard_ranges(ko, 0)


def _slice(w, s):
    d0, d1 = s.draft_rows
    t0, t1 = s.target_rows
    return dict(tl=w.target_logits[t0:t1], dl=w.draft_logits[d0:d1], ua=w.u_accept[d0:d1],
                ur=w.u_resample[t0:t1], ud=w.u_draft[d0:d1], T=w.temperature[s.b0:s.b1],
                ko=s.k_offsets)


def _batch():
    import workloads
    return workloads.make_case(B=13, k="ragged_1_10", V=300, dtype=workloads.BF16,
                               temperature="odd_greedy", sigma_d=0.7, seed=99, name="shard")


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    import oracle

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        w = _batch()
        s = shard.shard_for_rank(w.k_offsets, world, rank)
        x = _slice(w, s)
        ds = oracle.draft_sample(x["dl"], x["T"], x["ud"], x["ko"])
        vr = oracle.verify(x["tl"], x["dl"], ds.tokens, x["ua"], x["ur"], x["T"], x["ko"])
        assert ds.rc == 0 and vr.rc == 0
        mine = dict(draft=ds.tokens, tokens=vr.tokens, num=vr.num_accepted,
                    alpha=vr.accept_prob, z=vr.residual_mass)
        parts = [None] * world
        dist.all_gather_object(parts, mine)
        # the bench's timing reduction: max over ranks
        import torch
        t = torch.tensor([1.0 + rank])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        assert float(t) == float(world)
        if rank == 0:
            cat = {key: np.concatenate([p[key] for p in parts]) for key in mine}
            np.savez(os.path.join(out_dir, "gathered.npz"), **cat)
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_match_full_batch(tmp_path):
    import torch.multiprocessing as mp
    import oracle

    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = np.load(tmp_path / "gathered.npz")
    w = _batch()
    ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
    vr = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample,
                       w.temperature, w.k_offsets)
    assert np.array_equal(got["draft"], ds.tokens)
    assert np.array_equal(got["tokens"], vr.tokens)
    assert np.array_equal(got["num"], vr.num_accepted)
    assert np.array_equal(got["alpha"], vr.accept_prob, equal_nan=True)
    assert np.array_equal(got["z"], vr.residual_mass, equal_nan=True)
    # the split really put sequences on both ranks
    rr = shard.shard_ranges(w.k_offsets, world)
    assert all(b1 > b0 for b0, b1 in rr)
