"""GPU parity of the vocab-sharded verify (through the C ABI) against the
fp64 oracle run on the whole rows.

One GPU emulates G ranks in lockstep: each rank's three calls run on its own
column slice and workspace, and the two all-gathers become torch.stack over
the ranks' outputs (which is what an all-gather of them returns).  The final
element-wise maximum over ranks is the protocol's all-reduce.  Rules as for
the chain verify: tokens and counts bit-exact except sequences whose oracle
decision margin is <= 1e-5; greedy always exact.  Beyond parity: every rank
returns the same counts, and each sampled sequence is drawn by exactly one
rank.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from parity import compare_verify, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_61_gb300 as m
    m.lib()  # raises if the library is missing: no fallback
    return m


def lockstep(w, d, tokens, bounds):
    """The sharded verify of workload w over len(bounds) - 1 emulated ranks.
    Returns (tokens [R_t], num [B], per-rank token arrays)."""
    from speculative_decoding_verification_61_gb300.vocab_shard import VocabShardVerifier
    G = len(bounds) - 1
    code = 0 if w.dtype == workloads.F32 else 1
    tl, dl = d["target_logits"], d["draft_logits"]
    vs = [VocabShardVerifier(bounds, r, w.B, code) for r in range(G)]
    cols = [(tl[:, bounds[r]:bounds[r + 1]].contiguous(), dl[:, bounds[r]:bounds[r + 1]].contiguous())
            for r in range(G)]
    recs = [v.stats(t, q, tokens, d["temperature"], d["k_offsets"]) for v, (t, q) in zip(vs, cols)]
    all_recs = torch.stack(recs)
    outs = [v.decide(all_recs, d["u_accept"]) for v in vs]
    all_mass = torch.stack([o[2] for o in outs])
    toks = [v.draw(all_mass, d["u_resample"], o[0]) for v, o in zip(vs, outs)]
    torch.cuda.synchronize()
    nums = [o[1].cpu().numpy() for o in outs]
    for r in range(1, G):
        assert np.array_equal(nums[r], nums[0]), f"rank {r} took other decisions"
    per_rank = np.stack([t.cpu().numpy() for t in toks])
    return per_rank.max(axis=0), nums[0], per_rank


def check_one_owner(w, per_rank, num):
    """Each sampled, valid sequence's drawn slot holds a token on exactly one
    rank (-1 on the others); every other slot is equal on all ranks."""
    G = per_rank.shape[0]
    for b in range(w.B):
        k0, k1 = int(w.k_offsets[b]), int(w.k_offsets[b + 1])
        o = k0 + b
        sl = slice(o, k1 + b + 1)
        n = int(num[b])
        if n >= 0 and w.temperature[b] > 0:
            slot = per_rank[:, o + n]
            assert (slot >= 0).sum() == 1, (b, slot)
            rest = np.delete(per_rank[:, sl], n, axis=1)
        else:
            rest = per_rank[:, sl]
        assert (rest == rest[0]).all(), b
    return G


def oracle_tokens(w):
    ods = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets, nthreads=oracle.cores())
    return np.where(ods.tokens < 0, 0, ods.tokens).astype(np.int32)


def run_case(sv, w, bounds, seq_list=None):
    d = to_device(w)
    toks = oracle_tokens(w)
    got, num, per_rank = lockstep(w, d, torch.from_numpy(toks).cuda(), bounds)
    check_one_owner(w, per_rank, num)
    ora = oracle.verify(w.target_logits, w.draft_logits, toks, w.u_accept, w.u_resample, w.temperature,
                        w.k_offsets, seq_list=seq_list, nthreads=oracle.cores())
    assert ora.rc == 0
    flagged = compare_verify(w, got, num, None, ora, seq_list=seq_list)
    print(f"[vocab-shard parity] {w.name}: G={len(bounds) - 1}, {flagged} flagged, mean accepted {num.mean():.3f}")
    return got, num


def even(V, G):
    from speculative_decoding_verification_61_gb300.vocab_shard import even_bounds
    return even_bounds(V, G, 8)


KS = [0, 1, 2, 3, 5, 8, 13, 21, 32, 4, 7, 1]
CASES = [
    (dict(B=12, k=KS, V=20000, dtype="bf16", temperature=1.0), [0, 5000, 5008, 20000]),  # an 8-column shard
    (dict(B=12, k=KS, V=20000, dtype="f32", temperature=0.8), [0, 9996, 20000]),
    (dict(B=16, k="ragged_1_10", V=40008, dtype="bf16", temperature="odd_greedy",
          sigma_d="uniform_0.2_1.5"), "even5"),
    (dict(B=9, k=4, V=8, dtype="f32", temperature=1.0), [0, 4, 8]),                       # tiny vocabulary
    (dict(B=9, k=3, V=16, dtype="bf16", temperature=0.5), [0, 8, 16]),
    (dict(B=5, k=6, V=131072, dtype="bf16", temperature=0.05), "even8"),                   # sharp
    (dict(B=5, k=6, V=65536, dtype="f32", temperature=4.0), "even3"),                      # flat
    (dict(B=40, k=2, V=2056, dtype="bf16", temperature=1.0, sigma_d=3.0), "even4"),        # low acceptance
    (dict(B=40, k=6, V=3000, dtype="f32", temperature=1.0, sigma_d=0.05), "even2"),        # high acceptance
    (dict(B=7, k=5, V=4096, dtype="bf16", temperature=1.0), [0, 4096]),                    # one rank
    (dict(B=20, k="ragged_1_10", V=2048, dtype="bf16", temperature="odd_greedy"), "even16"),  # 16 ranks of 128 columns
    (dict(B=10, k="ragged_1_10", V=4096, dtype="bf16", temperature="odd_greedy"), "even64"),  # the most ranks: 64 of 64 columns
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_vocab_shard_parity_cases(sv, case):
    spec, bounds = CASES[case]
    w = workloads.make_case(seed=700 + case, **spec)
    if isinstance(bounds, str):
        bounds = even(w.V, int(bounds[4:]))
    run_case(sv, w, bounds)


def test_one_rank_equals_chain_verify(sv):
    """With G = 1 the sharded path reads the same rows as spec_verify: the
    decisions agree exactly wherever the oracle's margin is not tiny."""
    w = workloads.make_case(B=24, k="ragged_1_10", V=32000, dtype="bf16", temperature="odd_greedy", seed=71)
    d = to_device(w)
    toks = torch.from_numpy(oracle_tokens(w)).cuda()
    got, num, _ = lockstep(w, d, toks, [0, w.V])
    ct, cn = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, d["u_accept"], d["u_resample"],
                            d["temperature"], d["k_offsets"])
    ora = oracle.verify(w.target_logits, w.draft_logits, toks.cpu().numpy(), w.u_accept, w.u_resample,
                        w.temperature, w.k_offsets)
    compare_verify(w, got, num, None, ora)
    compare_verify(w, ct.cpu().numpy(), cn.cpu().numpy(), None, ora)
    assert np.array_equal(num, cn.cpu().numpy())


@pytest.mark.parametrize("G", [2, 8])
def test_vocab_shard_full_size_workload(sv, G):
    """The 512-sequence ragged workload (V = 128256, bf16) split over G ranks:
    the ownership and agreement checks on every sequence, oracle parity on
    a sample of 96 sequences (the oracle is slow at this V)."""
    w = workloads.make_config(5)
    rng = np.random.default_rng(G)
    seqs = np.sort(rng.choice(w.B, size=96, replace=False)).astype(np.int32)
    run_case(sv, w, even(w.V, G), seq_list=seqs)


def test_vocab_shard_data_errors(sv):
    """Data errors found in one rank's columns mark the sequence on every
    rank; a row that is -inf in one rank's columns only is valid."""
    w = workloads.make_case(B=8, k=3, V=4096, dtype="f32", temperature=1.0, seed=91)
    tl, dl = w.target_logits.copy(), w.draft_logits.copy()
    temp = w.temperature.copy()
    temp[7] = 0.0
    toks = oracle_tokens(workloads.Workload(**{**w.__dict__, "temperature": temp}))
    o = lambda b: int(w.k_offsets[b]) + b  # first target row of b
    tl[o(1) + 1, 3000] = np.nan        # NaN in rank 1's columns
    dl[int(w.k_offsets[2]) + 0, 100] = np.inf   # +inf in a draft row, rank 0's columns
    tl[o(3) + 0, :2048] = -np.inf      # -inf on rank 0 only: still a distribution
    tl[o(4) + 2, :] = -np.inf          # -inf everywhere: no distribution
    toks[int(w.k_offsets[5]) + 1] = 4096   # token outside [0, V)
    temp[6] = np.nan                   # bad temperature
    tl[o(7) + 1, 10] = np.nan          # greedy row with NaN
    w2 = workloads.Workload(**{**w.__dict__, "target_logits": tl, "draft_logits": dl, "temperature": temp})
    d = to_device(w2)
    got, num, per_rank = lockstep(w2, d, torch.from_numpy(toks).cuda(), [0, 2048, 4096])
    ora = oracle.verify(tl, dl, toks, w.u_accept, w.u_resample, temp, w.k_offsets)
    for b in (1, 2, 4, 5, 6, 7):
        assert ora.num_accepted[b] == -1 and num[b] == -1, b
    assert num[3] >= 0
    compare_verify(w2, got, num, None, ora)
    for b in (1, 2, 4, 5, 6, 7):
        k0, k1 = int(w.k_offsets[b]), int(w.k_offsets[b + 1])
        assert (per_rank[:, k0 + b:k1 + b + 1] == -1).all(), b


def test_vocab_shard_runs_of_rowless_sequences(sv):
    """Runs of sequences with a bad temperature (no rows streamed) between
    rows of one chunk per rank (G = 8 ranks of 1024 columns): every rank's
    streaming pass steps over them, the rest equal the oracle's outputs."""
    w = workloads.make_case(B=300, k="ragged_1_10", V=8192, dtype="bf16", temperature="odd_greedy", seed=93)
    temp = w.temperature.copy()
    bad = np.zeros(w.B, dtype=bool)
    for start in range(2, w.B, 61):
        bad[start:start + 30] = True
    bad[w.B - 20:] = True
    temp[bad] = -1.0
    w2 = workloads.Workload(**{**w.__dict__, "temperature": temp})
    got, num = run_case(sv, w2, even(w2.V, 8))
    assert (num[bad] == -1).all() and (num[~bad] >= 0).all()


def test_vocab_shard_invalid_offsets_fail_on_device(sv):
    from speculative_decoding_verification_61_gb300.vocab_shard import VocabShardVerifier
    w = workloads.make_case(B=4, k=3, V=2048, dtype="bf16", seed=5)
    d = to_device(w)
    ko = d["k_offsets"].clone()
    ko[2] = ko[1] + 33  # k_1 = 33 > SPEC_MAX_K
    bounds = [0, 1024, 2048]
    vs = [VocabShardVerifier(bounds, r, w.B, 1) for r in range(2)]
    toks = torch.zeros(w.rows_draft, dtype=torch.int32, device="cuda")
    cols = [(d["target_logits"][:, a:b].contiguous(), d["draft_logits"][:, a:b].contiguous())
            for a, b in zip(bounds[:-1], bounds[1:])]
    recs = [v.stats(t, q, toks, d["temperature"], ko) for v, (t, q) in zip(vs, cols)]
    _, num, mass = vs[0].decide(torch.stack(recs), d["u_accept"])
    # with caller outputs: the tokens stay untouched, every count is -1
    from speculative_decoding_verification_61_gb300 import spec_shard_decide
    out_t = torch.full((w.rows_target,), 77, dtype=torch.int32, device="cuda")
    _, num2, _ = spec_shard_decide(cols[0][0], cols[0][1], torch.stack(recs), toks, d["u_accept"], d["temperature"],
                                   ko, bounds, 0, vs[0].workspace, out_tokens=out_t)
    torch.cuda.synchronize()
    assert (num.cpu().numpy() == -1).all() and (num2.cpu().numpy() == -1).all()
    assert (out_t.cpu().numpy() == 77).all()
    assert (mass.cpu().numpy() == 0).all()
    assert sv.workspace_status(vs[0].workspace, clear=True) == -1
    assert sv.workspace_status(vs[0].workspace) == 0


def test_verify_vocab_sharded_nccl_world_of_one(sv, tmp_path):
    """The torch.distributed protocol itself (all-gathers and the MAX
    all-reduce over NCCL) on a group of one rank."""
    import torch.distributed as dist
    from speculative_decoding_verification_61_gb300.vocab_shard import VocabShardVerifier, verify_vocab_sharded
    w = workloads.make_case(B=16, k="ragged_1_10", V=16000, dtype="bf16", temperature="odd_greedy", seed=13)
    d = to_device(w)
    toks_np = oracle_tokens(w)
    toks = torch.from_numpy(toks_np).cuda()
    store = dist.FileStore(str(tmp_path / "store"), 1)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        v = VocabShardVerifier([0, w.V], 0, w.B, 1)
        got, num = verify_vocab_sharded(v, d["target_logits"], d["draft_logits"], toks, d["u_accept"],
                                        d["u_resample"], d["temperature"], d["k_offsets"])
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    ora = oracle.verify(w.target_logits, w.draft_logits, toks_np, w.u_accept, w.u_resample, w.temperature,
                        w.k_offsets)
    compare_verify(w, got.cpu().numpy(), num.cpu().numpy(), None, ora)


def test_vocab_shard_statistical_marginal(sv):
    """2^14 copies of one sequence (k = 1, V = 64, low acceptance so that most
    tokens come from the residual) split over three uneven ranks: the first
    emitted token follows p (chi-square), whichever rank drew it."""
    from scipy.special import softmax
    from scipy.stats import chisquare
    calls, B, V = 4, 4096, 64
    rng = np.random.default_rng(17)
    t = (rng.standard_normal(V) * 1.5).astype(np.float32)
    dr = (t + rng.standard_normal(V) * 1.5).astype(np.float32)
    bounds = [0, 24, 40, 64]
    urng = np.random.Generator(np.random.Philox(33))
    first = []
    for _ in range(calls):
        w = workloads.Workload(name="shared_seq", B=B, V=V, dtype="f32",
                               k_offsets=np.arange(B + 1, dtype=np.int32), temperature=np.ones(B, np.float32),
                               target_logits=np.tile(t, (2 * B, 1)), draft_logits=np.tile(dr, (B, 1)),
                               u_accept=workloads.uniforms(urng, B), u_resample=workloads.uniforms(urng, 2 * B),
                               u_draft=workloads.uniforms(urng, B))
        d = to_device(w)
        toks = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"])
        got, num, per_rank = lockstep(w, d, toks, bounds)
        check_one_owner(w, per_rank, num)
        first.append(got.reshape(B, 2)[:, 0])
    first = np.concatenate(first)
    p0 = softmax(t.astype(np.float64))
    counts = np.bincount(first, minlength=V)
    e = p0 * len(first)
    keep = e > 5
    c2 = np.append(counts[keep], counts[~keep].sum()).astype(np.float64)
    e2 = np.append(e[keep], e[~keep].sum())
    _, pval = chisquare(c2, e2 * c2.sum() / e2.sum())
    assert pval > 1e-4
    # the draws really came from every rank
    owners = {int(np.searchsorted(bounds, x, side="right")) - 1 for x in first}
    assert owners == {0, 1, 2}
