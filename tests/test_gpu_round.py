"""GPU tests of the fused round: draft sampling that keeps each draft row's
normaliser (spec_draft_sample_lse), verify that takes it instead of
re-reading the draft rows (spec_verify_lse), and both in one call
(spec_round).  All through the C ABI.

  * against the separate calls (spec_draft_sample, spec_verify): equal bit
    for bit, aux outputs included, since both derive the normaliser from
    the same partial sums;
  * against the fp64 oracle: the draft normalisers within the lse
    tolerance, and the verify outputs under the usual parity rules, on the
    full-size workloads.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import workloads
from parity import compare_draft, compare_verify, rtol_for, to_device

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
    dict(B=12, k=[0, 1, 2, 3, 5, 8, 13, 21, 32, 4, 7, 1], V=20000, dtype="bf16", temperature=1.0),
    dict(B=16, k="ragged_1_10", V=40008, dtype="bf16", temperature="odd_greedy",
         sigma_d="uniform_0.2_1.5"),
    dict(B=12, k=[0, 1, 2, 3, 5, 8, 13, 21, 32, 4, 7, 1], V=20000, dtype="f32", temperature=0.8),
    dict(B=9, k=4, V=8, dtype="f32", temperature=1.0),
    dict(B=40, k=2, V=2056, dtype="bf16", temperature=1.0, sigma_d=3.0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_calls_equal_separate_calls(sv, case):
    w = workloads.make_case(seed=300 + case, **CASES[case])
    d = to_device(w)
    args = (d["u_accept"], d["u_resample"], d["temperature"], d["k_offsets"])
    toks = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"])
    t0, n0, a0 = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, *args, aux=True)

    toks1, lse2 = sv.spec_draft_sample_lse(d["draft_logits"], d["temperature"], d["u_draft"],
                                           d["k_offsets"])
    assert torch.equal(toks1, toks)
    t1, n1, a1 = sv.spec_verify_lse(d["target_logits"], d["draft_logits"], lse2, toks, *args, aux=True)
    torch.cuda.synchronize()
    assert torch.equal(t1, t0) and torch.equal(n1, n0)
    for key in ("accept_prob", "residual_mass", "lse_target", "lse_draft"):
        x, y = a0[key].cpu().numpy(), a1[key].cpu().numpy()
        assert np.array_equal(x, y, equal_nan=True), key

    toks2, t2, n2 = sv.spec_round(d["target_logits"], d["draft_logits"], d["u_draft"], *args)
    torch.cuda.synchronize()
    assert torch.equal(toks2, toks) and torch.equal(t2, t0) and torch.equal(n2, n0)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fused_verify_matches_oracle(sv, cfg):
    """The oracle's draft tokens are verified with the GPU's draft
    normalisers; the normalisers themselves are checked against the
    oracle's draft-row log-sum-exp."""
    w = workloads.make_config(cfg)
    d = to_device(w)
    ods = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets,
                              nthreads=oracle.cores())
    gtok, lse2 = sv.spec_draft_sample_lse(d["draft_logits"], d["temperature"], d["u_draft"],
                                          d["k_offsets"])
    compare_draft(w, gtok.cpu().numpy(), ods)
    lse = lse2.cpu().numpy() * math.log(2.0)
    sampled_rows = np.repeat(w.temperature > 0, w.k)
    assert np.isnan(lse[~sampled_rows]).all()
    np.testing.assert_allclose(lse[sampled_rows], ods.lse[sampled_rows], rtol=rtol_for(w), atol=1e-6)

    toks = torch.from_numpy(ods.tokens).cuda()
    gt, gn, ga = sv.spec_verify_lse(d["target_logits"], d["draft_logits"], lse2, toks, d["u_accept"],
                                    d["u_resample"], d["temperature"], d["k_offsets"], aux=True)
    torch.cuda.synchronize()
    ora = oracle.verify(w.target_logits, w.draft_logits, ods.tokens, w.u_accept, w.u_resample,
                        w.temperature, w.k_offsets, nthreads=oracle.cores())
    compare_verify(w, gt.cpu().numpy(), gn.cpu().numpy(), {k: v.cpu().numpy() for k, v in ga.items()},
                   ora)


def test_bad_normaliser_marks_only_its_sequence(sv):
    w = workloads.make_case(B=6, k=3, V=4096, dtype="bf16", seed=41)
    d = to_device(w)
    toks, lse2 = sv.spec_draft_sample_lse(d["draft_logits"], d["temperature"], d["u_draft"],
                                          d["k_offsets"])
    args = (toks, d["u_accept"], d["u_resample"], d["temperature"], d["k_offsets"])
    t0, n0 = sv.spec_verify_lse(d["target_logits"], d["draft_logits"], lse2, *args)
    bad = lse2.clone()
    bad[2 * 3 + 0] = float("nan")   # sequence 2, position 0
    bad[4 * 3 + 2] = float("inf")   # sequence 4, position 2
    t1, n1 = sv.spec_verify_lse(d["target_logits"], d["draft_logits"], bad, *args)
    torch.cuda.synchronize()
    n0, n1, t0, t1 = (x.cpu().numpy() for x in (n0, n1, t0, t1))
    assert n1[2] == -1 and n1[4] == -1
    assert (t1[2 * 4:3 * 4] == -1).all() and (t1[4 * 4:5 * 4] == -1).all()
    keep = [0, 1, 3, 5]
    assert (n1[keep] == n0[keep]).all()
    for b in keep:
        assert (t1[b * 4:(b + 1) * 4] == t0[b * 4:(b + 1) * 4]).all()



def test_shutdown_frees_and_calls_allocate_again():
    """spec_shutdown frees the library-owned workspace and staging buffer;
    the next calls allocate them again and give the same outputs."""
    import speculative_decoding_verification_61_gb300 as sv
    w = workloads.make_case(B=16, k="ragged_1_10", V=20000, dtype="bf16", temperature="odd_greedy", seed=61)
    d = to_device(w)
    args = (d["target_logits"], d["draft_logits"], d["u_draft"], d["u_accept"], d["u_resample"], d["temperature"],
            d["k_offsets"])
    a = [x.clone() for x in sv.spec_round(*args)]
    h = lambda x: x.cpu().pin_memory()  # noqa: E731
    ah = sv.spec_round_host(*(h(x) for x in args))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    sv.shutdown()
    assert torch.cuda.mem_get_info()[0] > free0  # the buffers went back to the device
    b = sv.spec_round(*args)
    bh = sv.spec_round_host(*(h(x) for x in args))
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    for x, y in zip(ah, bh):
        assert torch.equal(x, y)
    for x, y in zip(a, ah):
        assert torch.equal(x.cpu(), y)


def test_graft_entry_smoke(sv):
    """The one-call smoke check of the package entry (one small draft sample
    and verify on cuda:0, compared with the oracle) runs clean."""
    import importlib.util
    import os
    spec = importlib.util.spec_from_file_location(
        "graft_entry", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "__graft_entry__.py"))
    entry = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(entry)
    entry.smoke()
