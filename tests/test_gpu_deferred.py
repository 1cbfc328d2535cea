"""GPU parity of the deferred epilogue (batches of 128 sequences or more).
Up to two sequences per resident streaming CTA (912 on a 152-SM GPU),
decide_stream_kernel decides and lists the rejected positions and streams
the listed row pairs in one launch; larger batches take resolve_kernel, then
resid_stream_kernel; resid_draw_kernel draws in both.  Against the fp64
oracle on shapes the full-size workloads do not cover: fp32 rows, a batch
with no rejection at all (all greedy; all accepted), many rejections, ragged
k with k = 0, data errors, the fused round and a caller workspace.  The
thresholds are checked by verifying the same sequences as a 127- and a
128-sequence batch, and as a 900- and a 1000-sequence batch."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from parity import compare_verify, gpu_verify, run_and_compare, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_61_gb300 as m
    m.lib()  # raises if the library is missing: no fallback
    return m


CASES = [
    dict(B=130, k=3, V=4096, dtype="f32", temperature=1.0, sigma_d=3.0),          # most positions rejected
    dict(B=160, k=4, V=2056, dtype="bf16", temperature=0.0),                      # all greedy: no pair
    dict(B=128, k=6, V=3000, dtype="f32", temperature=1.0, sigma_d=0.0),          # q = p: all accepted, no pair
    dict(B=200, k=[i % 11 for i in range(200)], V=16000, dtype="bf16", temperature=0.8),  # ragged, k = 0 included
    dict(B=256, k="ragged_1_10", V=40008, dtype="bf16", temperature="odd_greedy", sigma_d="uniform_0.2_1.5"),
    dict(B=300, k=[i % 33 for i in range(300)], V=2056, dtype="bf16", temperature=1.0, sigma_d=0.0),  # k 0..32, all accepted
    dict(B=300, k=[32 - i % 33 for i in range(300)], V=2056, dtype="f32", temperature="odd_greedy", sigma_d=2.5),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_deferred_epilogue_matches_the_oracle(sv, case):
    w = workloads.make_case(seed=500 + case, **CASES[case])
    rep = run_and_compare(w)
    if case == 2:
        assert rep["mean_accepted"] == 6.0  # q = p accepts every drafted token
    if case == 5:
        # q = p: every sequence accepts all k drafts and draws its bonus
        # token at position k (up to 32, the last u_resample slot)
        assert rep["mean_accepted"] == float(np.mean([i % 33 for i in range(300)]))


def test_deferred_data_errors_mark_only_their_sequence(sv):
    w = workloads.make_case(B=140, k=3, V=4096, dtype="f32", seed=509, temperature="odd_greedy", sigma_d=2.0)
    tl, dl = w.target_logits.copy(), w.draft_logits.copy()
    temp = w.temperature.copy()
    toks = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets).tokens.copy()
    tl[5 * 4 + 1, 9] = np.nan          # greedy sequence 5: NaN in a target row
    dl[8 * 3 + 2, 30] = np.inf         # sampled sequence 8: +inf in a draft row
    toks[12 * 3 + 0] = -3              # sequence 12: token out of range
    temp[20] = np.inf                  # sequence 20: bad temperature
    tl[30 * 4 + 3, :] = -np.inf        # sequence 30: bonus row entirely -inf
    w2 = workloads.Workload(**{**w.__dict__, "target_logits": tl, "draft_logits": dl, "temperature": temp})
    d = to_device(w2)
    gt, gn, ga = gpu_verify(d, torch.from_numpy(toks).cuda(), aux=True)
    ora = oracle.verify(tl, dl, toks, w.u_accept, w.u_resample, temp, w.k_offsets)
    gn = gn.cpu().numpy()
    for b in (5, 8, 12, 20, 30):
        assert ora.num_accepted[b] == -1 and gn[b] == -1, b
    compare_verify(w2, gt.cpu().numpy(), gn, {k: v.cpu().numpy() for k, v in ga.items()}, ora)


def test_threshold_batches_agree(sv):
    """The first 127 sequences verified as their own batch (one-kernel
    epilogue) and inside a 128-sequence batch (deferred epilogue) give the
    oracle's outputs; accept counts agree exactly between the two."""
    w = workloads.make_case(B=128, k="ragged_1_10", V=12000, dtype="bf16", seed=511, sigma_d=1.0)
    ods = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
    ora = oracle.verify(w.target_logits, w.draft_logits, ods.tokens, w.u_accept, w.u_resample, w.temperature,
                        w.k_offsets)
    d = to_device(w)
    toks = torch.from_numpy(ods.tokens).cuda()
    t128, n128 = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, d["u_accept"], d["u_resample"],
                                d["temperature"], d["k_offsets"])
    B1 = 127
    R_d, R_t = int(w.k_offsets[B1]), int(w.k_offsets[B1]) + B1
    t127, n127 = sv.spec_verify(d["target_logits"][:R_t], d["draft_logits"][:R_d], toks[:R_d],
                                d["u_accept"][:R_d], d["u_resample"][:R_t], d["temperature"][:B1],
                                d["k_offsets"][:B1 + 1].contiguous())
    torch.cuda.synchronize()
    compare_verify(w, t128.cpu().numpy(), n128.cpu().numpy(), None, ora)
    assert torch.equal(n128[:B1], n127)
    sub = workloads.Workload(**{**w.__dict__, "B": B1, "k_offsets": w.k_offsets[:B1 + 1],
                                "temperature": w.temperature[:B1]})
    compare_verify(sub, t127.cpu().numpy(), n127.cpu().numpy(), None, ora, seq_list=range(B1))


def test_deferred_round_and_caller_workspace(sv):
    """spec_round (the target pass streaming beside the draft draws) equals
    spec_draft_sample + spec_verify bit for bit at B >= 128, and a caller
    workspace gives the library workspace's outputs."""
    w = workloads.make_case(B=192, k="ragged_1_10", V=24000, dtype="bf16", seed=512, temperature="odd_greedy")
    d = to_device(w)
    args = (d["u_accept"], d["u_resample"], d["temperature"], d["k_offsets"])
    toks = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"])
    t0, n0 = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, *args)
    rt, rn, rd = [torch.empty_like(x) for x in (t0, n0, toks)]
    sv.spec_round(d["target_logits"], d["draft_logits"], d["u_draft"], *args, out_draft_tokens=rd,
                  out_tokens=rt, out_num_accepted=rn)
    ws = torch.zeros(sv.workspace_bytes(w.B, w.V, sv.BF16), dtype=torch.uint8, device="cuda")
    t1, n1 = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, *args, workspace=ws)
    t2, n2 = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, *args, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(rd, toks) and torch.equal(rt, t0) and torch.equal(rn, n0)
    assert torch.equal(t1, t0) and torch.equal(n1, n0) and torch.equal(t2, t0) and torch.equal(n2, n0)
    assert sv.workspace_status(ws) == 0
    ora = oracle.verify(w.target_logits, w.draft_logits, toks.cpu().numpy(), w.u_accept, w.u_resample,
                        w.temperature, w.k_offsets)
    compare_verify(w, t0.cpu().numpy(), n0.cpu().numpy(), None, ora)


def test_large_batch_forms_agree(sv):
    """The first 900 sequences verified as their own batch (one launch for
    decisions and residual stream) and inside a 1000-sequence batch
    (decisions, then the residual stream, as two launches) give the oracle's
    outputs; tokens and accept counts agree exactly between the two."""
    w = workloads.make_case(B=1000, k="ragged_1_10", V=4104, dtype="bf16", seed=513, temperature="odd_greedy",
                            sigma_d=1.5)
    ods = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
    ora = oracle.verify(w.target_logits, w.draft_logits, ods.tokens, w.u_accept, w.u_resample, w.temperature,
                        w.k_offsets)
    d = to_device(w)
    toks = torch.from_numpy(ods.tokens).cuda()
    tbig, nbig = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, d["u_accept"], d["u_resample"],
                                d["temperature"], d["k_offsets"])
    B1 = 900
    R_d, R_t = int(w.k_offsets[B1]), int(w.k_offsets[B1]) + B1
    tpre, npre = sv.spec_verify(d["target_logits"][:R_t], d["draft_logits"][:R_d], toks[:R_d],
                                d["u_accept"][:R_d], d["u_resample"][:R_t], d["temperature"][:B1],
                                d["k_offsets"][:B1 + 1].contiguous())
    torch.cuda.synchronize()
    compare_verify(w, tbig.cpu().numpy(), nbig.cpu().numpy(), None, ora)
    assert torch.equal(nbig[:B1], npre) and torch.equal(tbig[:R_t], tpre)
    kb = np.diff(w.k_offsets)[:B1]
    pairs = (npre.cpu().numpy() < kb) & (w.temperature[:B1] > 0)  # sampled sequences with a rejection
    assert int(pairs.sum()) > 100
    sub = workloads.Workload(**{**w.__dict__, "B": B1, "k_offsets": w.k_offsets[:B1 + 1],
                                "temperature": w.temperature[:B1]})
    compare_verify(sub, tpre.cpu().numpy(), npre.cpu().numpy(), None, ora, seq_list=range(B1))
