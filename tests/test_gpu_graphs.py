"""The entry points under CUDA graph capture (GPU).

A serving loop replays the verify step as a captured graph. Every call here
is captured once after an eager warm-up (the library-owned workspace is
allocated then, never during capture), replayed several times, and must
give the eager call's outputs bit for bit: nothing in the library may
depend on host state that capture freezes, or synchronise the stream.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads
from parity import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_61_gb300 as m
    m.lib()  # raises if the library is missing: no fallback
    return m


def replay_equals_eager(run, outs, reps=3):
    """run() writes into the tensors in outs; eager first, then captured."""
    run()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for o in outs:
        o.fill_(-7)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        run()
    for _ in range(reps):
        for o in outs:
            o.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, eager):
            assert torch.equal(a, b)


def test_spec_round_and_verify_under_capture(sv):
    w = workloads.make_case(B=48, k="ragged_1_10", V=32000, dtype="bf16", temperature="odd_greedy", seed=21)
    d = to_device(w)
    toks = torch.empty(w.rows_draft, dtype=torch.int32, device="cuda")
    out_t = torch.empty(w.rows_target, dtype=torch.int32, device="cuda")
    out_n = torch.empty(w.B, dtype=torch.int32, device="cuda")
    args = (d["target_logits"], d["draft_logits"], d["u_draft"], d["u_accept"], d["u_resample"], d["temperature"],
            d["k_offsets"])
    replay_equals_eager(lambda: sv.spec_round(*args, out_draft_tokens=toks, out_tokens=out_t, out_num_accepted=out_n),
                        [toks, out_t, out_n])
    # spec_verify on the round's tokens, and the two-call form
    vt = torch.empty_like(out_t)
    vn = torch.empty_like(out_n)
    replay_equals_eager(lambda: sv.spec_verify(d["target_logits"], d["draft_logits"], toks, d["u_accept"],
                                               d["u_resample"], d["temperature"], d["k_offsets"], out_tokens=vt,
                                               out_num_accepted=vn), [vt, vn])
    assert torch.equal(vt, out_t) and torch.equal(vn, out_n)


@pytest.mark.parametrize("B", [160, 1000])
def test_deferred_epilogue_under_capture(sv, B):
    """Batches of 128 sequences or more take the deferred epilogue: one launch
    for decisions and residual stream up to two sequences per resident CTA
    (B = 160), two launches beyond (B = 1000 on a 152-SM GPU).  Both replay
    bit for bit."""
    w = workloads.make_case(B=B, k="ragged_1_10", V=8192, dtype="bf16", temperature="odd_greedy", seed=23 + B,
                            sigma_d=1.5)
    d = to_device(w)
    toks = torch.empty(w.rows_draft, dtype=torch.int32, device="cuda")
    out_t = torch.empty(w.rows_target, dtype=torch.int32, device="cuda")
    out_n = torch.empty(w.B, dtype=torch.int32, device="cuda")
    args = (d["target_logits"], d["draft_logits"], d["u_draft"], d["u_accept"], d["u_resample"], d["temperature"],
            d["k_offsets"])
    replay_equals_eager(lambda: sv.spec_round(*args, out_draft_tokens=toks, out_tokens=out_t, out_num_accepted=out_n),
                        [toks, out_t, out_n])
    vt = torch.empty_like(out_t)
    vn = torch.empty_like(out_n)
    replay_equals_eager(lambda: sv.spec_verify(d["target_logits"], d["draft_logits"], toks, d["u_accept"],
                                               d["u_resample"], d["temperature"], d["k_offsets"], out_tokens=vt,
                                               out_num_accepted=vn), [vt, vn])
    assert torch.equal(vt, out_t) and torch.equal(vn, out_n)
    assert int((vn.cpu() < torch.from_numpy(np.diff(w.k_offsets))).sum()) > B // 4  # residual draws happened


def test_tree_verify_under_capture(sv):
    w = workloads.make_tree_case(B=20, shape=[3, 2], V=8192, dtype="bf16", temperature=1.0, seed=31)
    t = lambda a: (torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)  # noqa: E731
                   if a.dtype == np.uint16 else torch.from_numpy(np.ascontiguousarray(a))).cuda()
    d = {k: t(getattr(w, k)) for k in ("target_logits", "draft_logits", "node_offsets", "parent", "u_accept",
                                       "u_resample", "u_draft", "temperature")}
    toks = sv.spec_tree_draft_sample(d["draft_logits"], d["node_offsets"], d["parent"], d["temperature"],
                                     d["u_draft"])
    toks = torch.where(toks < 0, torch.zeros_like(toks), toks)
    outs = [torch.empty(w.nodes, dtype=torch.int32, device="cuda"), torch.empty(w.B, dtype=torch.int32, device="cuda"),
            torch.empty(w.B, dtype=torch.int32, device="cuda")]
    replay_equals_eager(lambda: sv.spec_tree_verify(d["target_logits"], d["draft_logits"], d["node_offsets"],
                                                    d["parent"], toks, d["u_accept"], d["u_resample"],
                                                    d["temperature"], out_tokens=outs[0], out_num_accepted=outs[1],
                                                    out_last_node=outs[2]), outs)


def test_vocab_shard_rank_under_capture(sv):
    from speculative_decoding_verification_61_gb300.vocab_shard import VocabShardVerifier
    w = workloads.make_case(B=24, k="ragged_1_10", V=16000, dtype="bf16", temperature=1.0, seed=41)
    d = to_device(w)
    toks = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"])
    bounds = [0, 8000, 16000]
    vs = [VocabShardVerifier(bounds, r, w.B, 1) for r in range(2)]
    cols = [(d["target_logits"][:, a:b].contiguous(), d["draft_logits"][:, a:b].contiguous())
            for a, b in zip(bounds, bounds[1:])]
    recs = torch.stack([v.stats(tl, dl, toks, d["temperature"], d["k_offsets"]) for v, (tl, dl) in zip(vs, cols)])
    outs = [v.decide(recs, d["u_accept"]) for v in vs]
    mass = torch.stack([o[2] for o in outs])
    rec0 = torch.empty_like(recs[0])
    tok0, num0, mass0 = (torch.empty_like(x) for x in outs[0])
    from speculative_decoding_verification_61_gb300 import spec_shard_decide, spec_shard_draw, spec_shard_stats

    def rank0():
        spec_shard_stats(cols[0][0], cols[0][1], toks, d["temperature"], d["k_offsets"], bounds, 0, vs[0].workspace,
                         out_stats=rec0)
        spec_shard_decide(cols[0][0], cols[0][1], recs, toks, d["u_accept"], d["temperature"], d["k_offsets"],
                          bounds, 0, vs[0].workspace, out_tokens=tok0, out_num_accepted=num0, out_mass=mass0)
        spec_shard_draw(cols[0][0], cols[0][1], mass, d["u_resample"], d["k_offsets"], bounds, 0, vs[0].workspace,
                        tok0)
    replay_equals_eager(rank0, [rec0, tok0, num0, mass0])
    assert torch.equal(rec0, recs[0])
