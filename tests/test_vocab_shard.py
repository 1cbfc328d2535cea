"""The vocab-sharded verify's exchange protocol on CPU ranks (gloo).

verify_vocab_sharded runs its all-gathers and the final MAX all-reduce over
real torch.distributed ranks here; the three device steps of each rank are
replaced by NumpyShardSteps, an fp64 stand-in with the library's record
formats (on GPUs, VocabShardVerifier runs them in the CUDA library; that
path's parity is in test_gpu_vocab_shard.py).  The ranks' joint result must
be the oracle's verify on the whole rows, and every rank must return it.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

from speculative_decoding_verification_61_gb300 import vocab_shard

LOG2E = 1.4426950408889634


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_even_bounds():
    assert vocab_shard.even_bounds(128256, 8) == [16032 * r for r in range(9)]
    b = vocab_shard.even_bounds(40008, 5)
    assert b[0] == 0 and b[-1] == 40008 and all((y - x) % 8 == 0 and y > x for x, y in zip(b, b[1:]))
    assert vocab_shard.even_bounds(16, 2, 8) == [0, 8, 16]
    with pytest.raises(ValueError):
        vocab_shard.even_bounds(16, 3, 8)   # fewer blocks of 8 than ranks
    with pytest.raises(ValueError):
        vocab_shard.even_bounds(100, 2, 8)  # V not a multiple of 8


class NumpyShardSteps:
    """One rank's three steps in fp64 numpy (test stand-in for the device):
    records [R_t + R_d, 4] int32 (m, s, zx as float32 bits, arg), masses
    [B, 2] float64, the same rules as the library's kernels."""

    def __init__(self, bounds, rank):
        self.bounds, self.rank = list(bounds), rank
        self.G = len(bounds) - 1
        self.v0, self.v1 = bounds[rank], bounds[rank + 1]

    def stats(self, target_shard, draft_shard, draft_tokens, temperature, k_offsets):
        import torch
        self.t = target_shard.numpy().astype(np.float64)
        self.d = draft_shard.numpy().astype(np.float64)
        self.x, self.T, self.ko = draft_tokens.numpy(), temperature.numpy(), k_offsets.numpy()
        B = len(self.T)
        R_d = int(self.ko[B])
        R_t = R_d + B
        rec = np.zeros((R_t + R_d, 4), np.int32)
        f = rec.view(np.float32)
        f[:, 0], f[:, 1], rec[:, 3] = -np.inf, np.nan, -1
        for b in range(B):
            T, k = float(self.T[b]), int(self.ko[b + 1] - self.ko[b])
            if not (T >= 0 and np.isfinite(T)):
                continue
            rows = [(int(self.ko[b]) + b + i, self.t[int(self.ko[b]) + b + i], i) for i in range(k + 1)]
            if T > 0:
                rows += [(R_t + int(self.ko[b]) + i, self.d[int(self.ko[b]) + i], i) for i in range(k)]
            for r, z, i in rows:
                if T == 0:
                    if np.isnan(z).any():
                        rec[r, 3] = -1
                    else:
                        rec[r, 3] = self.v0 + int(np.argmax(z))
                    f[r, 0], f[r, 1], f[r, 2] = z.max(), 0.0, 0.0
                    continue
                y = z * (LOG2E / T)
                if np.isnan(y).any() or np.isposinf(y).any():
                    m, s = -np.inf, np.nan
                else:
                    m = y.max()
                    s = np.exp2(y - m).sum() if m > -np.inf else 0.0
                f[r, 0], f[r, 1], rec[r, 3] = m, s, 0
                x = int(self.x[int(self.ko[b]) + i]) if i < k else -1
                f[r, 2] = z[x - self.v0] if self.v0 <= x < self.v1 else 0.0
        return torch.from_numpy(rec)

    def _combine(self, recs):  # recs [G, 4] int32 -> (M, S, ok)
        f = recs.view(np.float32).astype(np.float64)
        m, s = f[:, 0], f[:, 1]
        M = m.max()
        if np.isnan(s).any() or not np.isfinite(M):
            return M, 0.0, False
        S = float(sum(s[g] * 2.0 ** (m[g] - M) for g in range(self.G) if m[g] > -np.inf))
        return M, S, S > 0 and np.isfinite(S)

    def decide(self, all_stats, u_accept):
        import torch
        A = all_stats.numpy()
        B = len(self.T)
        R_d = int(self.ko[B])
        R_t = R_d + B
        out = np.full(R_t, -1, np.int32)
        num = np.full(B, -1, np.int32)
        mass = np.zeros((B, 2))
        self.seq = [None] * B
        ua = u_accept.numpy()
        for b in range(B):
            T, k, ot, od = float(self.T[b]), int(self.ko[b + 1] - self.ko[b]), int(self.ko[b]) + b, int(self.ko[b])
            xs = self.x[od:od + k]
            if not (T >= 0 and np.isfinite(T)) or ((xs < 0) | (xs >= self.bounds[-1])).any():
                continue
            if T == 0:
                args = []
                for i in range(k + 1):
                    r = A[:, ot + i]
                    if (r[:, 3] < 0).any():
                        break
                    v = r.view(np.float32)[:, 0]
                    args.append(int(r[int(np.argmax(v)), 3]))  # first rank with the max: lowest column
                if len(args) < k + 1:
                    continue
                n = next((i for i in range(k) if xs[i] != args[i]), k)
                out[ot:ot + n], out[ot + n], num[b] = xs[:n], args[n], n
                continue
            owner = lambda x: int(np.searchsorted(self.bounds, x, side="right")) - 1
            Mt, St, Lt, Ld, okk = [], [], [], [], True
            for i in range(k + 1):
                M, S, ok = self._combine(A[:, ot + i])
                okk &= ok
                Mt.append(M), St.append(S), Lt.append(M + np.log2(S) if ok else np.nan)
            for i in range(k):
                M, S, ok = self._combine(A[:, R_t + od + i])
                okk &= ok
                Ld.append(M + np.log2(S) if ok else np.nan)
            if not okk:
                continue
            n = k
            for i in range(k):
                g = owner(int(xs[i]))
                zt = float(A[g, ot + i].view(np.float32)[2])
                zd = float(A[g, R_t + od + i].view(np.float32)[2])
                c = LOG2E / T
                alpha = 0.0 if zt == -np.inf else 1.0 if zd == -np.inf else min(1.0, 2.0 ** ((zt * c - Lt[i]) - (zd * c - Ld[i])))
                if not ua[od + i] < alpha:
                    n = i
                    break
            out[ot:ot + n], num[b] = xs[:n], n
            c = LOG2E / T
            pw = np.exp2(self.t[ot + n] * c - Mt[n])
            if n < k:
                w = np.maximum(0.0, np.exp2(self.t[ot + n] * c - Lt[n]) - np.exp2(self.d[od + n] * c - Ld[n]))
            else:
                w = pw
            self.seq[b] = (ot + n, w, pw)
            mass[b] = w.sum(), pw.sum()
        return torch.from_numpy(out), torch.from_numpy(num), torch.from_numpy(mass)

    def draw(self, all_mass, u_resample, out_tokens):
        am = all_mass.numpy()
        ur = u_resample.numpy()
        out = out_tokens.numpy()
        for b, sq in enumerate(self.seq):
            if sq is None:
                continue
            slot, w, pw = sq
            col = 0 if am[:, b, 0].sum() > 0 else 1
            Z = am[:, b, col].sum()
            t = float(ur[slot]) * Z
            C, owner = 0.0, -1
            for g in range(self.G):
                if am[g, b, col] > 0 and C + am[g, b, col] > t:
                    owner = g
                    break
                C += am[g, b, col]
            if owner != self.rank:
                continue
            ww = w if col == 0 else pw
            cum = np.cumsum(ww)
            hit = np.flatnonzero((cum > t - C) & (ww > 0))
            out[slot] = self.v0 + int(hit[0] if hit.size else np.flatnonzero(ww > 0)[-1])
        return out_tokens


def _batch():
    import workloads
    return workloads.make_case(B=11, k="ragged_1_10", V=600, dtype=workloads.F32, temperature="odd_greedy",
                               sigma_d=0.7, seed=123, name="vocab_shard")


def _rank_main(rank, world, port, out_dir, bounds):
    import torch
    import torch.distributed as dist

    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w = _batch()
        ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
        toks = np.where(ds.tokens < 0, 0, ds.tokens).astype(np.int32)
        a, b = bounds[rank], bounds[rank + 1]
        steps = NumpyShardSteps(bounds, rank)
        got, num = vocab_shard.verify_vocab_sharded(
            steps, torch.from_numpy(np.ascontiguousarray(w.target_logits[:, a:b])),
            torch.from_numpy(np.ascontiguousarray(w.draft_logits[:, a:b])), torch.from_numpy(toks),
            torch.from_numpy(w.u_accept), torch.from_numpy(w.u_resample), torch.from_numpy(w.temperature),
            torch.from_numpy(w.k_offsets))
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), tokens=got.numpy(), num=num.numpy(), toks=toks)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("bounds", [[0, 296, 600], [0, 8, 400, 600]])
def test_gloo_ranks_match_whole_row_verify(tmp_path, bounds):
    import torch.multiprocessing as mp

    import oracle
    from parity import FLAG_MARGIN
    world = len(bounds) - 1
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path), bounds), nprocs=world, join=True)
    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    for r in range(1, world):
        assert np.array_equal(res[r]["tokens"], res[0]["tokens"])
        assert np.array_equal(res[r]["num"], res[0]["num"])
    w = _batch()
    ora = oracle.verify(w.target_logits, w.draft_logits, res[0]["toks"], w.u_accept, w.u_resample,
                        w.temperature, w.k_offsets)
    tok, num = res[0]["tokens"], res[0]["num"]
    compared = 0
    for b in range(w.B):
        if ora.num_accepted[b] >= 0 and ora.margin[b] <= FLAG_MARGIN:
            continue
        sl = slice(int(w.k_offsets[b]) + b, int(w.k_offsets[b + 1]) + b + 1)
        assert num[b] == ora.num_accepted[b], b
        assert (tok[sl] == ora.tokens[sl]).all(), (b, tok[sl], ora.tokens[sl])
        compared += 1
    assert compared >= w.B - 1
    # the draws really landed on several ranks
    assert len({int(np.searchsorted(bounds, t, side="right")) - 1 for t in tok[tok >= 0]}) > 1


def test_verify_vocab_sharded_checks_the_group():
    """The protocol refuses a verifier whose shards do not match the group."""
    import torch.distributed as dist
    store = dist.HashStore()
    dist.init_process_group("gloo", store=store, rank=0, world_size=1)
    try:
        steps = NumpyShardSteps([0, 8, 16], 0)
        with pytest.raises(ValueError):
            vocab_shard.verify_vocab_sharded(steps, *([None] * 7))
    finally:
        dist.destroy_process_group()
