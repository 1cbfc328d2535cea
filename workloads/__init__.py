"""Seeded synthetic inputs for the speculative-decoding verify step.

This module is the only code shared by the CPU oracle's tests and the CUDA
path.  It draws random numbers and lays them out; it computes none of the
method's arithmetic (no softmax, no acceptance test, no sampling).  Draft
tokens are therefore NOT produced here: they come from a draft-sampling
implementation (the oracle in tests, the CUDA `spec_draft_sample` in the
benchmark), fed with the uniforms `u_draft` drawn here.

Logit recipe (Zipf-like rows with Gaussian noise, the shape the verify step
sees from a real target/draft pair):

* target row:  z_t[v] = -a * ln(1 + pi_r(v)) + N(0, sigma_t^2), with pi_r a
  permutation of the vocabulary drawn per row: one random arrangement P of
  the vocabulary per workload, rotated by a random offset per row,
  pi_r(v) = P[(v + c_r) mod V].  Each row keeps its multiset of logits
  exactly Zipf + noise and puts its large logits at different token ids;
  rotations make 128K-wide rows cheap to draw.  make_case(perm="per_row")
  draws instead a fresh, independent permutation pi_r for every row (the
  workload text's wording taken literally), for parity cases;
* draft row i of a sequence: z_d = z_t(target row i of that sequence) +
  N(0, sigma_d^2);
* bf16 workloads are generated in fp32 and rounded to bf16 here
  (round-to-nearest-even on the fp32 bit pattern), so that both sides read
  identical bits.

Random streams: k_b (ragged batches) from the workload seed; then one
independent PCG64 stream per sequence (SeedSequence spawn), so a sequence's
logits do not depend on how many threads generate the batch.  Uniforms are
fp32 multiples of 2^-24 in [0, 1), drawn from a Philox generator in the
fixed order u_accept, u_resample, u_draft.

Layout (packed, ragged k per sequence):
  k_offsets [B+1] int32, exclusive prefix sum of k_b (k_offsets[0] = 0)
  target_logits [k_offsets[B] + B, V]  rows o_b .. o_b + k_b with o_b = k_offsets[b] + b
  draft_logits  [k_offsets[B], V]      rows k_offsets[b] .. k_offsets[b+1]-1
  u_accept [k_offsets[B]], u_resample [k_offsets[B] + B], u_draft [k_offsets[B]]
  temperature [B] fp32 (0 = greedy)
bf16 arrays are numpy uint16 holding the bf16 bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"

# The five workloads: (B, k or None for ragged 1..10, V, dtype, temperature
# rule, a, sigma_t, sigma_d rule).
CONFIGS = {
    1: dict(name="tiny_B4_k4_V1000_f32", B=4, k=4, V=1000, dtype=F32,
            temperature=1.0, a=1.1, sigma_t=1.0, sigma_d=0.5),
    2: dict(name="B8_k4_V32000_f32", B=8, k=4, V=32000, dtype=F32,
            temperature=1.0, a=1.1, sigma_t=1.0, sigma_d=0.5),
    3: dict(name="B64_k5_V128256_bf16_T0.7", B=64, k=5, V=128256, dtype=BF16,
            temperature=0.7, a=1.1, sigma_t=1.5, sigma_d=1.0),
    4: dict(name="B256_k8_V152064_bf16_half_greedy", B=256, k=8, V=152064,
            dtype=BF16, temperature="odd_greedy", a=1.1, sigma_t=1.0,
            sigma_d="uniform_0.2_1.5"),
    5: dict(name="B512_ragged_k1to10_V128256_bf16", B=512, k="ragged_1_10",
            V=128256, dtype=BF16, temperature=1.0, a=1.1, sigma_t=1.0,
            sigma_d=0.5),
}


@dataclass
class Workload:
    """One batch of verify-step inputs (host numpy arrays)."""

    name: str
    B: int
    V: int
    dtype: str
    k_offsets: np.ndarray          # int32 [B+1]
    temperature: np.ndarray        # float32 [B]
    target_logits: np.ndarray      # float32 or uint16(bf16 bits) [R_t, V]
    draft_logits: np.ndarray       # same dtype [R_d, V]
    u_accept: np.ndarray           # float32 [R_d]
    u_resample: np.ndarray         # float32 [R_t]
    u_draft: np.ndarray            # float32 [R_d]
    meta: dict = field(default_factory=dict)

    @property
    def k(self) -> np.ndarray:
        return np.diff(self.k_offsets)

    @property
    def rows_target(self) -> int:
        return int(self.k_offsets[-1]) + self.B

    @property
    def rows_draft(self) -> int:
        return int(self.k_offsets[-1])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    rounded = bits + np.uint32(0x7FFF) + lsb
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniforms(rng: np.random.Generator, n: int) -> np.ndarray:
    """n fp32 uniforms in [0, 1), each an exact multiple of 2^-24."""
    return (rng.integers(0, 1 << 24, size=n, dtype=np.int64).astype(np.float64)
            * (1.0 / (1 << 24))).astype(np.float32)


def make_case(B: int, k, V: int, dtype: str = F32, temperature=1.0, a: float = 1.1,
              sigma_t: float = 1.0, sigma_d=0.5, seed: int = 1234,
              uniform_seed: int = 0, name: str | None = None, perm: str = "rotated") -> Workload:
    """Build a workload.

    k: int (uniform), a sequence of per-sequence k_b, or "ragged_1_10".
    temperature: float (all sequences), a sequence, or "odd_greedy" (odd
      sequences T=0, even sequences T=1).
    sigma_d: float, or "uniform_0.2_1.5" (one sigma per draft row).
    perm: "rotated" (one arrangement per workload, rotated per row) or
      "per_row" (an independent random permutation for every target row).
    """
    assert perm in ("rotated", "per_row")
    ss = np.random.SeedSequence(seed)
    ss_k, ss_layout, ss_seq = ss.spawn(3)
    if isinstance(k, str):
        assert k == "ragged_1_10"
        ks = np.random.default_rng(ss_k).integers(1, 11, size=B, dtype=np.int64)
    elif np.isscalar(k):
        ks = np.full(B, int(k), dtype=np.int64)
    else:
        ks = np.asarray(k, dtype=np.int64)
        assert ks.shape == (B,)
    k_offsets = np.zeros(B + 1, dtype=np.int32)
    k_offsets[1:] = np.cumsum(ks)
    R_d = int(k_offsets[-1])
    R_t = R_d + B

    if isinstance(temperature, str):
        assert temperature == "odd_greedy"
        temp = np.where(np.arange(B) % 2 == 1, 0.0, 1.0).astype(np.float32)
    elif np.isscalar(temperature):
        temp = np.full(B, float(temperature), dtype=np.float32)
    else:
        temp = np.asarray(temperature, dtype=np.float32)
        assert temp.shape == (B,)

    base = (-a * np.log1p(np.arange(V, dtype=np.float64))).astype(np.float32)
    arranged = base[np.random.default_rng(ss_layout).permutation(V)]
    odt = np.uint16 if dtype == BF16 else np.float32
    assert dtype in (BF16, F32)
    zt_out = np.empty((R_t, V), dtype=odt)
    zd_out = np.empty((R_d, V), dtype=odt)
    seq_seeds = ss_seq.spawn(B)

    def store(dst, row):
        dst[:] = round_to_bf16_bits(row) if dtype == BF16 else row

    def one_sequence(b):
        rng = np.random.default_rng(seq_seeds[b])
        k_b = int(ks[b])
        t0, d0 = int(k_offsets[b]) + b, int(k_offsets[b])
        shifts = rng.integers(0, V, size=k_b + 1)
        if isinstance(sigma_d, str):
            assert sigma_d == "uniform_0.2_1.5"
            sig = rng.uniform(0.2, 1.5, size=k_b)
        else:
            sig = np.full(k_b, float(sigma_d))
        row = np.empty(V, dtype=np.float32)
        for i in range(k_b + 1):
            if perm == "per_row":
                row[:] = base[rng.permutation(V)]
            else:
                c = int(shifts[i])
                row[:V - c] = arranged[c:]
                row[V - c:] = arranged[:c]
            row += rng.standard_normal(V, dtype=np.float32) * np.float32(sigma_t)
            store(zt_out[t0 + i], row)
            if i < k_b:
                d = row + rng.standard_normal(V, dtype=np.float32) * np.float32(sig[i])
                store(zd_out[d0 + i], d)

    workers = max(1, min(32, os.cpu_count() or 1))
    if B > 1 and workers > 1:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one_sequence, range(B)))
    else:
        for b in range(B):
            one_sequence(b)
    zt, zd = zt_out, zd_out

    urng = np.random.Generator(np.random.Philox(uniform_seed))
    u_accept = uniforms(urng, R_d)
    u_resample = uniforms(urng, R_t)
    u_draft = uniforms(urng, R_d)
    return Workload(name=name or f"B{B}_V{V}_{dtype}", B=B, V=V, dtype=dtype,
                    k_offsets=k_offsets, temperature=temp, target_logits=zt,
                    draft_logits=zd, u_accept=u_accept, u_resample=u_resample,
                    u_draft=u_draft,
                    meta=dict(a=a, sigma_t=sigma_t, sigma_d=sigma_d, seed=seed,
                              uniform_seed=uniform_seed, perm=perm))


def make_config(cfg: int) -> Workload:
    """Workload number cfg (1..5) with its fixed seeds (logits: 1000+cfg,
    uniforms: 0)."""
    c = CONFIGS[cfg]
    return make_case(B=c["B"], k=c["k"], V=c["V"], dtype=c["dtype"],
                     temperature=c["temperature"], a=c["a"], sigma_t=c["sigma_t"],
                     sigma_d=c["sigma_d"], seed=1000 + cfg, uniform_seed=0,
                     name=c["name"])


def algorithmic_bytes(w: Workload, n_sampled: int | None = None) -> dict:
    """Bytes the verify step must move at minimum, by the accounting rule:
    every needed logit row read once (target rows; draft rows of sampled
    sequences only) plus one row-equivalent per sampled sequence for the
    resample.  Also the draft-sampling pass (every draft row once), and
    the verify pass that takes the draft rows' normalisers from it."""
    s = w.elem_bytes
    sampled = w.temperature > 0
    ks = w.k
    rows_needed = w.rows_target + int(ks[sampled].sum())
    n_s = int(sampled.sum()) if n_sampled is None else n_sampled
    small = (w.B + 1) * 4 + w.B * 4 + w.rows_draft * 4 * 2 + w.rows_target * 4 * 2 + w.B * 4
    verify = s * w.V * (rows_needed + n_s) + small
    draft = s * w.V * w.rows_draft + w.rows_draft * 4 * 2 + (w.B + 1) * 4 + w.B * 4
    # verify with the draft rows' normalisers given: target rows once, the
    # resample row-equivalent, and 8 bytes of normaliser per sampled draft row
    verify_lse = s * w.V * (w.rows_target + n_s) + 8 * int(ks[sampled].sum()) + small
    return dict(verify=int(verify), draft_sample=int(draft), verify_lse=int(verify_lse),
                rows_verified=int(w.rows_target + w.rows_draft),
                rows_needed=int(rows_needed), sampled_sequences=n_s)


def seq_rows(w: Workload, b: int):
    """(target row range, draft row range) of sequence b."""
    k0, k1 = int(w.k_offsets[b]), int(w.k_offsets[b + 1])
    return range(k0 + b, k1 + b + 1), range(k0, k1)


# ------------------------------------------------------------------ trees
@dataclass
class TreeWorkload:
    """One batch of tree-verify inputs (host numpy arrays).  Sequence b owns
    nodes node_offsets[b] .. node_offsets[b+1]-1, the first being its root;
    every node has a target row and a draft row (the distributions after the
    path to it; a leaf's draft row is part of the layout but not needed)."""

    name: str
    B: int
    V: int
    dtype: str
    node_offsets: np.ndarray       # int32 [B+1]
    parent: np.ndarray             # int32 [N], -1 for roots
    temperature: np.ndarray        # float32 [B]
    target_logits: np.ndarray      # [N, V]
    draft_logits: np.ndarray       # [N, V]
    u_accept: np.ndarray           # float32 [N]
    u_resample: np.ndarray         # float32 [N]
    u_draft: np.ndarray            # float32 [N]
    meta: dict = field(default_factory=dict)

    @property
    def nodes(self) -> int:
        return int(self.node_offsets[-1])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def internal(self) -> np.ndarray:
        """bool [N]: node has at least one child."""
        out = np.zeros(self.nodes, dtype=bool)
        out[self.parent[self.parent >= 0]] = True
        return out


def tree_shape(branching) -> np.ndarray:
    """Parent array (breadth-first order) of a full tree with the given
    number of children per node at each depth, e.g. [3, 2, 1]."""
    parent = [-1]
    level = [0]
    for m in branching:
        nxt = []
        for u in level:
            for _ in range(int(m)):
                parent.append(u)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.asarray(parent, dtype=np.int32)


def make_tree_case(B: int, shape, V: int, dtype: str = F32, temperature=1.0, a: float = 1.1,
                   sigma_t: float = 1.0, sigma_d: float = 0.5, seed: int = 4321,
                   uniform_seed: int = 0, name: str | None = None) -> TreeWorkload:
    """Build a tree workload.

    shape: a list of branching factors (one full tree for every sequence),
      "random_N" (per sequence a random recursive tree of 1..N nodes: node i
      hangs under a uniformly chosen earlier node), or a list of B parent
      arrays (local indices, -1 for the root).
    temperature: float, a sequence, or "odd_greedy".
    Rows follow the chain recipe: target row = Zipf slope a rotated per row +
    N(0, sigma_t^2); draft row = that target row + N(0, sigma_d^2).
    """
    ss = np.random.SeedSequence(seed)
    ss_shape, ss_layout, ss_seq = ss.spawn(3)
    if isinstance(shape, str):
        assert shape.startswith("random_")
        nmax = int(shape.split("_")[1])
        srng = np.random.default_rng(ss_shape)
        shapes = []
        for _ in range(B):
            n = int(srng.integers(1, nmax + 1))
            par = [-1] + [int(srng.integers(0, i)) for i in range(1, n)]
            shapes.append(np.asarray(par, dtype=np.int32))
    elif len(shape) == B and not np.isscalar(shape[0]):
        shapes = [np.asarray(s, dtype=np.int32) for s in shape]
    else:
        one = tree_shape(shape)
        shapes = [one] * B
    sizes = np.array([len(s) for s in shapes], dtype=np.int64)
    node_offsets = np.zeros(B + 1, dtype=np.int32)
    node_offsets[1:] = np.cumsum(sizes)
    N = int(node_offsets[-1])
    parent = np.empty(N, dtype=np.int32)
    for b, s in enumerate(shapes):
        g0 = int(node_offsets[b])
        parent[g0:g0 + len(s)] = np.where(s >= 0, s + g0, -1)

    if isinstance(temperature, str):
        assert temperature == "odd_greedy"
        temp = np.where(np.arange(B) % 2 == 1, 0.0, 1.0).astype(np.float32)
    elif np.isscalar(temperature):
        temp = np.full(B, float(temperature), dtype=np.float32)
    else:
        temp = np.asarray(temperature, dtype=np.float32)

    base = (-a * np.log1p(np.arange(V, dtype=np.float64))).astype(np.float32)
    arranged = base[np.random.default_rng(ss_layout).permutation(V)]
    odt = np.uint16 if dtype == BF16 else np.float32
    assert dtype in (BF16, F32)
    zt_out = np.empty((N, V), dtype=odt)
    zd_out = np.empty((N, V), dtype=odt)
    seq_seeds = ss_seq.spawn(B)

    def store(dst, row):
        dst[:] = round_to_bf16_bits(row) if dtype == BF16 else row

    def one_sequence(b):
        rng = np.random.default_rng(seq_seeds[b])
        g0, n = int(node_offsets[b]), int(sizes[b])
        shifts = rng.integers(0, V, size=n)
        row = np.empty(V, dtype=np.float32)
        for i in range(n):
            c = int(shifts[i])
            row[:V - c] = arranged[c:]
            row[V - c:] = arranged[:c]
            row += rng.standard_normal(V, dtype=np.float32) * np.float32(sigma_t)
            store(zt_out[g0 + i], row)
            d = row + rng.standard_normal(V, dtype=np.float32) * np.float32(sigma_d)
            store(zd_out[g0 + i], d)

    workers = max(1, min(32, os.cpu_count() or 1))
    if B > 1 and workers > 1:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one_sequence, range(B)))
    else:
        for b in range(B):
            one_sequence(b)

    urng = np.random.Generator(np.random.Philox(uniform_seed))
    u_accept = uniforms(urng, N)
    u_resample = uniforms(urng, N)
    u_draft = uniforms(urng, N)
    return TreeWorkload(name=name or f"tree_B{B}_N{N}_V{V}_{dtype}", B=B, V=V, dtype=dtype,
                        node_offsets=node_offsets, parent=parent, temperature=temp,
                        target_logits=zt_out, draft_logits=zd_out, u_accept=u_accept,
                        u_resample=u_resample, u_draft=u_draft,
                        meta=dict(a=a, sigma_t=sigma_t, sigma_d=sigma_d, seed=seed,
                                  uniform_seed=uniform_seed))


# the tree workload measured beside the chain workloads: 64 sequences, each a
# full tree of 3 / 2 / 1 children per depth (16 nodes), as a static
# Medusa/EAGLE-style candidate tree
TREE_CONFIG = dict(name="tree_B64_n16_b321_V128256_bf16", B=64, shape=[3, 2, 1], V=128256,
                   dtype=BF16, temperature=1.0, a=1.1, sigma_t=1.0, sigma_d=0.5)


def make_tree_config() -> TreeWorkload:
    c = dict(TREE_CONFIG)
    return make_tree_case(seed=2000, uniform_seed=0, **c)


def tree_algorithmic_bytes(w: TreeWorkload) -> int:
    """Bytes a tree verify must move at minimum: every node's target row and
    every internal node's draft row once (sampled sequences), plus one
    row-equivalent per sampled sequence for the residual or bonus draw."""
    s = w.elem_bytes
    internal = w.internal()
    seq_of = np.repeat(np.arange(w.B), np.diff(w.node_offsets))
    sampled = w.temperature[seq_of] > 0
    rows = w.nodes + int((internal & sampled).sum())
    return int(s * w.V * (rows + int((w.temperature > 0).sum())))
