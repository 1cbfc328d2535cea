"""GPU parity of the tree (multi-candidate) verify and tree drafting
(through the C ABI) against the fp64 oracle on seeded inputs.

Rules as for the chain verify: the accepted count, the node the walk ended
at and the emitted tokens are bit-exact, except for sequences whose oracle
decision margin is <= 1e-5 (counted, not compared); greedy is always exact.
Tokens come from the oracle's tree drafting, so that verify parity does not
depend on drafting margins; the GPU's drafting is compared separately.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from parity import FLAG_MARGIN

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_61_gb300 as m
    m.lib()  # raises if the library is missing: no fallback
    return m


def dev(a):
    x = torch.from_numpy(np.ascontiguousarray(a))
    return (x.view(torch.bfloat16) if a.dtype == np.uint16 else x).cuda()


def tree_inputs(w):
    return {k: dev(getattr(w, k)) for k in ("target_logits", "draft_logits", "node_offsets", "parent",
                                            "u_accept", "u_resample", "u_draft", "temperature")}


def compare_tree(w, tokens, got, ora):
    gt, gn, gl = (x.cpu().numpy() for x in got)
    flagged = 0
    for b in range(w.B):
        g0, g1 = int(w.node_offsets[b]), int(w.node_offsets[b + 1])
        if ora.num_accepted[b] >= 0 and ora.margin[b] <= FLAG_MARGIN:
            flagged += 1
            continue
        assert gn[b] == ora.num_accepted[b], (b, gn[b], ora.num_accepted[b])
        assert gl[b] == ora.last_node[b], (b, gl[b], ora.last_node[b])
        assert (gt[g0:g1] == ora.tokens[g0:g1]).all(), (b, gt[g0:g1], ora.tokens[g0:g1])
    return flagged


def run_tree_parity(sv, w):
    d = tree_inputs(w)
    od = oracle.tree_draft_sample(w.draft_logits, w.node_offsets, w.parent, w.temperature, w.u_draft,
                                  nthreads=oracle.cores())
    tokens = np.where(od.tokens < 0, 0, od.tokens).astype(np.int32)
    got = sv.spec_tree_verify(d["target_logits"], d["draft_logits"], d["node_offsets"], d["parent"],
                              dev(tokens), d["u_accept"], d["u_resample"], d["temperature"])
    torch.cuda.synchronize()
    ora = oracle.tree_verify(w.target_logits, w.draft_logits, w.node_offsets, w.parent, tokens, w.u_accept,
                             w.u_resample, w.temperature, nthreads=oracle.cores())
    assert ora.rc == 0
    flagged = compare_tree(w, tokens, got, ora)
    n = got[1].cpu().numpy()
    print(f"[tree parity] {w.name}: {w.B} sequences, {flagged} flagged, mean accepted {n.mean():.3f}")
    return got, ora


CASES = [
    dict(B=24, shape="random_8", V=4096, dtype="f32", temperature=1.0),
    dict(B=24, shape="random_12", V=20000, dtype="bf16", temperature="odd_greedy"),
    dict(B=16, shape=[3, 2, 1], V=40008, dtype="bf16", temperature=0.7),
    dict(B=32, shape=[4], V=3000, dtype="f32", temperature=1.0, sigma_d=3.0),   # four candidates, low acceptance
    dict(B=4, shape=[2, 2, 2, 2, 2], V=1000, dtype="f32", temperature=1.0),     # 63 nodes
    dict(B=16, shape=[1, 1, 1, 1], V=20000, dtype="bf16", temperature=1.0),     # a chain
    dict(B=9, shape="random_6", V=8, dtype="f32", temperature=1.0),              # tiny vocabulary
    dict(B=200, shape=[2, 2], V=4096, dtype="bf16", temperature=1.0, sigma_d=2.0),  # 400 CTAs: several waves of clusters
    dict(B=8, shape=[63], V=4096, dtype="f32", temperature=1.0, sigma_d=3.0),   # 64 nodes (the most): 63 candidates at the root
    dict(B=4096, shape=[2], V=64, dtype="bf16", temperature="odd_greedy"),      # the most sequences per call
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_tree_parity_cases(sv, case):
    w = workloads.make_tree_case(seed=500 + case, **CASES[case])
    run_tree_parity(sv, w)


def test_tree_full_size_workload(sv):
    """The benchmark's tree workload at full size, every sequence checked;
    its drafting on the GPU against the oracle's too."""
    w = workloads.make_tree_config()
    got, ora = run_tree_parity(sv, w)
    d = tree_inputs(w)
    gd = sv.spec_tree_draft_sample(d["draft_logits"], d["node_offsets"], d["parent"], d["temperature"],
                                   d["u_draft"]).cpu().numpy()
    od = oracle.tree_draft_sample(w.draft_logits, w.node_offsets, w.parent, w.temperature, w.u_draft,
                                  nthreads=oracle.cores())
    ok = od.margin > FLAG_MARGIN
    assert (gd[ok] == od.tokens[ok]).all()
    assert (gd[w.parent < 0] == -1).all()


def test_tree_draft_sample_parity(sv):
    w = workloads.make_tree_case(B=20, shape="random_10", V=12000, dtype="bf16", temperature="odd_greedy",
                                 seed=77)
    d = tree_inputs(w)
    gd = sv.spec_tree_draft_sample(d["draft_logits"], d["node_offsets"], d["parent"], d["temperature"],
                                   d["u_draft"]).cpu().numpy()
    od = oracle.tree_draft_sample(w.draft_logits, w.node_offsets, w.parent, w.temperature, w.u_draft)
    ok = od.margin > FLAG_MARGIN
    assert (gd[ok] == od.tokens[ok]).all()
    assert (gd[w.parent < 0] == -1).all()


def test_tree_runs_of_rowless_trees(sv):
    """Runs of trees with a bad temperature (no rows streamed; one run at the
    batch's end) between trees whose rows are one chunk, so that a ticket of
    the streaming passes lies many trees ahead: the drafting and the verify
    equal the oracle's outputs, and every row-less tree is -1."""
    w = workloads.make_tree_case(B=300, shape=[2, 2], V=4096, dtype="bf16", temperature=1.0, sigma_d=1.0,
                                 seed=590)
    temp = w.temperature.copy()
    bad = np.zeros(w.B, dtype=bool)
    for start in range(1, w.B, 53):
        bad[start:start + 25] = True
    bad[w.B - 15:] = True
    temp[bad] = -1.0
    w2 = workloads.TreeWorkload(**{**w.__dict__, "temperature": temp})
    d = tree_inputs(w2)
    gd = sv.spec_tree_draft_sample(d["draft_logits"], d["node_offsets"], d["parent"], d["temperature"],
                                   d["u_draft"]).cpu().numpy()
    od = oracle.tree_draft_sample(w2.draft_logits, w2.node_offsets, w2.parent, temp, w2.u_draft)
    ok = od.margin > FLAG_MARGIN
    assert (gd[ok] == od.tokens[ok]).all()
    got, ora = run_tree_parity(sv, w2)
    n = got[1].cpu().numpy()
    assert (n[bad] == -1).all() and (ora.num_accepted[bad] == -1).all() and (n[~bad] >= 0).all()


def test_tree_data_errors(sv):
    w = workloads.make_tree_case(B=6, shape=[2, 1], V=4096, dtype="f32", seed=88)
    tl = w.target_logits.copy()
    parent = w.parent.copy()
    temp = w.temperature.copy()
    od = oracle.tree_draft_sample(w.draft_logits, w.node_offsets, w.parent, w.temperature, w.u_draft)
    tokens = np.where(od.tokens < 0, 0, od.tokens).astype(np.int32)
    n = 5  # nodes per tree
    parent[1 * n + 2] = 1 * n + 3      # sequence 1: a node's parent comes after it
    tokens[2 * n + 1] = 4096           # sequence 2: token out of range
    tl[3 * n + 0, 5] = np.nan          # sequence 3: NaN in the root's target row
    temp[4] = -1.0                     # sequence 4: bad temperature
    w2 = workloads.TreeWorkload(**{**w.__dict__, "target_logits": tl, "parent": parent, "temperature": temp})
    d = tree_inputs(w2)
    got = sv.spec_tree_verify(d["target_logits"], d["draft_logits"], d["node_offsets"], d["parent"], dev(tokens),
                              d["u_accept"], d["u_resample"], d["temperature"])
    ora = oracle.tree_verify(tl, w.draft_logits, w.node_offsets, parent, tokens, w.u_accept, w.u_resample, temp)
    gn = got[1].cpu().numpy()
    for b in (1, 2, 3, 4):
        assert ora.num_accepted[b] == -1 and gn[b] == -1, b
    compare_tree(w2, tokens, got, ora)
    # an invalid node_offsets array fails the whole call on the device
    no = w.node_offsets.copy()
    no[3] = no[2]  # an empty sequence
    out_t = torch.full((w.nodes,), 77, dtype=torch.int32, device="cuda")
    _, gn2, _ = sv.spec_tree_verify(d["target_logits"], d["draft_logits"], dev(no), d["parent"], dev(tokens),
                                    d["u_accept"], d["u_resample"], dev(w.temperature), out_tokens=out_t)
    torch.cuda.synchronize()
    assert (gn2.cpu().numpy() == -1).all()
    assert (out_t.cpu().numpy() == 77).all()
    assert sv.workspace_status(clear=True) == -1
    assert sv.workspace_status() == 0


def test_tree_statistical_marginal(sv):
    """2^14 copies of one tree (a root with three candidates) sharing p and
    q, V = 64, in four calls of 4096: the first emitted token follows p_root
    (chi-square)."""
    from scipy.special import softmax
    from scipy.stats import chisquare
    calls, B, V = 4, 4096, 64
    rng = np.random.default_rng(9)
    t = (rng.standard_normal((4, V)) * 1.5).astype(np.float32)
    dr = (t + rng.standard_normal((4, V)) * 1.0).astype(np.float32)
    shape = np.array([-1, 0, 0, 0], np.int32)
    parent = np.where(np.tile(shape, B) >= 0, np.tile(shape, B) + np.repeat(np.arange(B) * 4, 4), -1).astype(np.int32)
    urng = np.random.Generator(np.random.Philox(21))
    first = []
    for _ in range(calls):
        w = workloads.TreeWorkload(name="shared_tree", B=B, V=V, dtype="f32",
                                   node_offsets=(np.arange(B + 1) * 4).astype(np.int32), parent=parent,
                                   temperature=np.ones(B, np.float32), target_logits=np.tile(t, (B, 1)),
                                   draft_logits=np.tile(dr, (B, 1)), u_accept=workloads.uniforms(urng, 4 * B),
                                   u_resample=workloads.uniforms(urng, 4 * B),
                                   u_draft=workloads.uniforms(urng, 4 * B))
        d = tree_inputs(w)
        toks = sv.spec_tree_draft_sample(d["draft_logits"], d["node_offsets"], d["parent"], d["temperature"],
                                         d["u_draft"])
        toks = torch.where(toks < 0, torch.zeros_like(toks), toks)
        gt, gn, _ = sv.spec_tree_verify(d["target_logits"], d["draft_logits"], d["node_offsets"], d["parent"],
                                        toks, d["u_accept"], d["u_resample"], d["temperature"])
        first.append(gt.cpu().numpy().reshape(B, 4)[:, 0])
    first = np.concatenate(first)
    p0 = softmax(t[0].astype(np.float64))
    counts = np.bincount(first, minlength=V)
    e = p0 * len(first)
    keep = e > 5
    c2 = np.append(counts[keep], counts[~keep].sum()).astype(np.float64)
    e2 = np.append(e[keep], e[~keep].sum())
    _, pval = chisquare(c2, e2 * c2.sum() / e2.sum())
    assert pval > 1e-4
