"""Failure detection on the GPU without a GPU fault: the library's bounded
waits are made to run out (an mbarrier nothing arrives at, a meeting
counter nothing completes, a residual pair nobody lists), report
SPEC_ERR_TIMEOUT through the status word, and leave the context usable for
the next call."""
from __future__ import annotations

import pytest

import oracle
import workloads
from parity import compare_verify, gpu_draft_sample, gpu_verify, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_61_gb300 as m
    m.lib()  # raises if the library is missing: no fallback
    return m


def test_bounded_waits_give_up_and_report_timeout(sv):
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")  # the 256-byte counters block
    sv.selfcheck_wait_timeout(ws)
    torch.cuda.synchronize()  # about 6 s: three waits of 2 s
    assert sv.workspace_status(ws) == -4  # SPEC_ERR_TIMEOUT
    assert int(ws[8]) == 7  # all three waits gave up
    assert int(ws[9]) == 0  # the meeting counter was put back
    assert sv.workspace_status(ws, clear=True) == -4 and sv.workspace_status(ws) == 0
    # the context is still usable: a verify afterwards matches the oracle
    w = workloads.make_case(B=6, k=4, V=2000, dtype="f32", seed=5)
    d = to_device(w)
    toks = gpu_draft_sample(d)
    gt, gn, _ = gpu_verify(d, toks)
    torch.cuda.synchronize()
    ora = oracle.verify(w.target_logits, w.draft_logits, toks.cpu().numpy(), w.u_accept, w.u_resample,
                        w.temperature, w.k_offsets)
    compare_verify(w, gt.cpu().numpy(), gn.cpu().numpy(), None, ora)


def test_timed_out_workspace_reports_every_sequence_as_an_error(sv):
    """While a workspace's status word holds SPEC_ERR_TIMEOUT (a bounded wait
    gave up, so its partials may be of any age), verify and draft-sampling
    calls on it mark every sequence and row -1 instead of giving outputs that
    look valid; once the status is cleared the same calls match the
    library-owned workspace's results again."""
    w = workloads.make_case(B=6, k=4, V=2000, dtype="f32", seed=7, temperature="odd_greedy")
    d = to_device(w)
    toks = gpu_draft_sample(d)
    ref_t, ref_n, _ = gpu_verify(d, toks)
    ws = torch.zeros(sv.workspace_bytes(w.B, w.V, sv.F32), dtype=torch.uint8, device="cuda")
    sv.selfcheck_wait_timeout(ws)  # records SPEC_ERR_TIMEOUT in ws (about 6 s)
    args = (d["u_accept"], d["u_resample"], d["temperature"], d["k_offsets"])
    gt, gn = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, *args, workspace=ws)
    gd = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"], workspace=ws)
    torch.cuda.synchronize()
    assert sv.workspace_status(ws) == -4
    assert (gn == -1).all() and (gt == -1).all() and (gd == -1).all()
    assert sv.workspace_status(ws, clear=True) == -4
    gt, gn = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, *args, workspace=ws)
    gd = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"], workspace=ws)
    torch.cuda.synchronize()
    assert sv.workspace_status(ws) == 0
    assert torch.equal(gt, ref_t) and torch.equal(gn, ref_n) and torch.equal(gd, toks)
