"""Vocab-sharded verify over a process group (one rank per GPU).

Each rank holds the logits of its own vocabulary columns [V_r, V_{r+1}) for
every target and draft row, as a tensor-parallel LM head leaves them.  One
verify is three library calls per rank with two all-gathers between them and
an element-wise maximum at the end:

    records = stats(own columns)                  spec_shard_stats
    all_records = all_gather(records)             [G, R_t + R_d, 4] int32
    tokens, num, mass = decide(all_records)       spec_shard_decide
    all_mass = all_gather(mass)                   [G, B, 2] float64
    tokens = draw(all_mass)                       spec_shard_draw
    all_reduce(tokens, MAX)                       the drawn token from its owner

Every rank takes the same decisions (the records are combined in rank
order on each), so num_accepted needs no exchange; the drawn token is -1
on every rank but the one whose columns hold it.  The result is that of
spec_verify on the full rows, up to the order of floating-point sums.

This module is host logic only: the three steps run in the CUDA library
(VocabShardVerifier), the exchanges in torch.distributed (NCCL on GPUs).
"""
from __future__ import annotations

from . import _binding


def even_bounds(V: int, G: int, multiple: int = 8) -> list[int]:
    """Shard bounds [0, V_1, ..., V] with G nearly equal widths, each width a
    multiple of `multiple` (8 keeps bf16 and fp32 rows 16-byte aligned)."""
    if G < 1 or V % multiple:
        raise ValueError(f"V={V} must be a multiple of {multiple} and G >= 1")
    units = V // multiple
    if units < G:
        raise ValueError(f"V={V} has fewer than G={G} blocks of {multiple} columns")
    return [(units * r // G) * multiple for r in range(G + 1)]


class VocabShardVerifier:
    """One rank's side of a vocab-sharded verify: the three steps on this
    rank's columns, with the call's inputs kept between them.  The
    workspace (the library's state between the steps) is allocated once and
    reused by every verify with at most `max_B` sequences."""

    def __init__(self, shard_bounds, rank: int, max_B: int, dtype: int, device="cuda"):
        self.bounds = [int(x) for x in shard_bounds]
        self.G = len(self.bounds) - 1
        if not 0 <= rank < self.G:
            raise ValueError(f"rank {rank} outside [0, {self.G})")
        self.rank = rank
        self.Vs = self.bounds[rank + 1] - self.bounds[rank]
        self.max_B = max_B
        self.dtype = dtype
        self.workspace = _binding.shard_workspace(max_B, self.Vs, dtype, device)
        self._call = None

    def stats(self, target_shard, draft_shard, draft_tokens, temperature, k_offsets, stream=None):
        B = temperature.numel()
        if B > self.max_B:
            raise ValueError(f"B={B} exceeds the workspace's {self.max_B}")
        if target_shard.shape[-1] != self.Vs or draft_shard.shape[-1] != self.Vs:
            raise ValueError(f"shards must have {self.Vs} columns")
        self._call = dict(target_shard=target_shard, draft_shard=draft_shard, draft_tokens=draft_tokens,
                          temperature=temperature, k_offsets=k_offsets)
        return _binding.spec_shard_stats(target_shard, draft_shard, draft_tokens, temperature, k_offsets,
                                         self.bounds, self.rank, self.workspace, stream=stream)

    def decide(self, all_stats, u_accept, stream=None):
        c = self._call
        return _binding.spec_shard_decide(c["target_shard"], c["draft_shard"], all_stats, c["draft_tokens"],
                                          u_accept, c["temperature"], c["k_offsets"], self.bounds, self.rank,
                                          self.workspace, stream=stream)

    def draw(self, all_mass, u_resample, out_tokens, stream=None):
        c = self._call
        return _binding.spec_shard_draw(c["target_shard"], c["draft_shard"], all_mass, u_resample,
                                        c["k_offsets"], self.bounds, self.rank, self.workspace, out_tokens,
                                        stream=stream)


def _all_gather(t, group):
    import torch
    import torch.distributed as dist
    parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def verify_vocab_sharded(verifier, target_shard, draft_shard, draft_tokens, u_accept, u_resample, temperature,
                         k_offsets, group=None):
    """One vocab-sharded verify on this rank (collective over `group`, whose
    rank order must be the shard order).  `verifier` is this rank's
    VocabShardVerifier.  Returns (out_tokens [R_t] int32, out_num_accepted
    [B] int32), equal on every rank."""
    import torch.distributed as dist
    if dist.get_world_size(group) != verifier.G or dist.get_rank(group) != verifier.rank:
        raise ValueError("the group's size and rank must match the verifier's shards")
    records = verifier.stats(target_shard, draft_shard, draft_tokens, temperature, k_offsets)
    all_records = _all_gather(records, group)
    tokens, num, mass = verifier.decide(all_records, u_accept)
    all_mass = _all_gather(mass, group)
    tokens = verifier.draw(all_mass, u_resample, tokens)
    dist.all_reduce(tokens, op=dist.ReduceOp.MAX, group=group)
    return tokens, num
