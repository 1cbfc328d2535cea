"""Shared parity helpers: run the CUDA path (through the C ABI binding) and
the fp64 oracle on the same seeded inputs and compare them.

Rules (the verify step's contract):
  * tokens and accept counts bit-exact, except for sequences whose oracle
    decision margin is <= 1e-5 (a uniform within 1e-5 of an accept threshold
    alpha_i, or of a CDF boundary C_v / Z of the draw that was taken); those
    are counted as flagged and not compared;
  * greedy sequences and arg-max draws are always exact (no flagging);
  * accept probabilities alpha, residual mass Z and per-row log-sum-exp
    within 1e-5 relative for fp32 logits, 2e-3 for bf16 logits.
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads

FLAG_MARGIN = 1e-5


def rtol_for(w) -> float:
    return 1e-5 if w.dtype == workloads.F32 else 2e-3


def to_device(w, device="cuda"):
    import torch
    def t(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            x = x.view(torch.bfloat16)
        return x.to(device)
    return dict(target_logits=t(w.target_logits), draft_logits=t(w.draft_logits),
                u_accept=t(w.u_accept), u_resample=t(w.u_resample), u_draft=t(w.u_draft),
                temperature=t(w.temperature), k_offsets=t(w.k_offsets))


def gpu_draft_sample(d, stream=None):
    from speculative_decoding_verification_61_gb300 import spec_draft_sample
    return spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"],
                             stream=stream)


def gpu_verify(d, draft_tokens, aux=True):
    from speculative_decoding_verification_61_gb300 import spec_verify
    return spec_verify(d["target_logits"], d["draft_logits"], draft_tokens, d["u_accept"],
                       d["u_resample"], d["temperature"], d["k_offsets"], aux=aux)


def compare_draft(w, gpu_tokens, ora):
    """Draft-sample parity: exact except flagged sampled rows.  Returns
    (flagged rows, flagged rows whose token still matches)."""
    g = np.asarray(gpu_tokens)
    flagged = ora.margin <= FLAG_MARGIN
    mism = (g != ora.tokens) & ~flagged
    assert not mism.any(), (f"{mism.sum()} draft rows differ, first at "
                            f"{np.flatnonzero(mism)[:5]}: gpu {g[mism][:5]} oracle {ora.tokens[mism][:5]}")
    return int(flagged.sum()), int((flagged & (g == ora.tokens)).sum())


def compare_verify(w, gtok, gnum, gaux, ora, seq_list=None, stats=None):
    """Verify parity; returns the number of flagged sequences.  `stats`, if
    given, receives the flagged count and how many flagged sequences still
    match exactly."""
    gtok, gnum = np.asarray(gtok), np.asarray(gnum)
    seqs = range(w.B) if seq_list is None else seq_list
    rtol = rtol_for(w)
    flagged = flagged_match = 0
    for b in seqs:
        k0, k1 = int(w.k_offsets[b]), int(w.k_offsets[b + 1])
        o = k0 + b
        sl = slice(o, k1 + b + 1)
        if ora.num_accepted[b] >= 0 and ora.margin[b] <= FLAG_MARGIN:
            flagged += 1
            flagged_match += int(gnum[b] == ora.num_accepted[b] and (gtok[sl] == ora.tokens[sl]).all())
            continue
        assert gnum[b] == ora.num_accepted[b], (b, gnum[b], ora.num_accepted[b])
        assert (gtok[sl] == ora.tokens[sl]).all(), (b, gtok[sl], ora.tokens[sl])
    if stats is not None:
        stats.update(flagged=flagged, flagged_match=flagged_match)
    if gaux is None:
        return flagged
    ap, z = np.asarray(gaux["accept_prob"]), np.asarray(gaux["residual_mass"])
    lt, ld = np.asarray(gaux["lse_target"]), np.asarray(gaux["lse_draft"])
    for b in seqs:
        if ora.num_accepted[b] < 0 or w.temperature[b] == 0:
            continue
        k0, k1 = int(w.k_offsets[b]), int(w.k_offsets[b + 1])
        o = k0 + b
        if k1 > k0:
            np.testing.assert_allclose(ap[k0:k1], ora.accept_prob[k0:k1], rtol=rtol, atol=1e-7,
                                       err_msg=f"alpha of sequence {b}")
            np.testing.assert_allclose(ld[k0:k1], ora.lse_draft[k0:k1], rtol=rtol, atol=1e-6,
                                       err_msg=f"draft lse of sequence {b}")
        np.testing.assert_allclose(lt[o:k1 + b + 1], ora.lse_target[o:k1 + b + 1], rtol=rtol,
                                   atol=1e-6, err_msg=f"target lse of sequence {b}")
        if ora.num_accepted[b] < k1 - k0 and not np.isnan(ora.residual_mass[b]):
            np.testing.assert_allclose(z[b], ora.residual_mass[b], rtol=rtol, atol=1e-9,
                                       err_msg=f"residual mass of sequence {b}")
    return flagged


def run_and_compare(w, nthreads=None, seq_list=None, check_draft=True):
    """Full round on the GPU (draft sample, then verify on the oracle's
    draft tokens) and on the oracle.  Returns a small report dict."""
    import torch
    nthreads = nthreads or oracle.cores()
    d = to_device(w)
    ods = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets,
                              nthreads=nthreads)
    rep = {}
    if check_draft and w.rows_draft:
        gds = gpu_draft_sample(d).cpu().numpy()
        rep["draft_flagged"], rep["draft_flagged_match"] = compare_draft(w, gds, ods)
    tokens = torch.from_numpy(ods.tokens).cuda()
    gtok, gnum, gaux = gpu_verify(d, tokens, aux=True)
    torch.cuda.synchronize()
    gaux = {k: v.cpu().numpy() for k, v in gaux.items()}
    ora = oracle.verify(w.target_logits, w.draft_logits, ods.tokens, w.u_accept, w.u_resample,
                        w.temperature, w.k_offsets, seq_list=seq_list, nthreads=nthreads)
    st = {}
    rep["verify_flagged"] = compare_verify(w, gtok.cpu().numpy(), gnum.cpu().numpy(), gaux, ora,
                                           seq_list=seq_list, stats=st)
    rep["verify_flagged_match"] = st["flagged_match"]
    rep["sequences"] = w.B if seq_list is None else len(seq_list)
    rep["mean_accepted"] = float(np.mean(gnum.cpu().numpy()))
    print(f"[parity] {w.name}: {rep}")
    return rep
