"""The allocation-free verify entry point (spec_verify_noalloc).

It exists for callers that cannot allocate device memory while they verify:
serving loops that keep allocation off the hot path, and runtimes whose
memory pool owns the whole GPU.  Its scratch memory is a fixed array inside
the library, so these tests check that it
gives exactly the outputs of spec_verify (all outputs are integers: token
ids and accept counts, compared exactly, as every GPU parity test does
outside flagged margins), on two calls in a row (the array keeps the first
call's contents), and that batches too large for the array are refused.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_61_gb300 import build
    build.build()
    import speculative_decoding_verification_61_gb300 as m
    m.lib()
    return m


def _device(w):
    def t(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(torch.bfloat16) if a.dtype == np.uint16 else x).cuda()
    return {k: t(getattr(w, k)) for k in ("target_logits", "draft_logits", "u_accept", "u_resample",
                                         "u_draft", "temperature", "k_offsets")}


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc_call(sv, d, toks, V, dtype):
    """Calls the entry point through the C ABI directly (ctypes)."""
    R_t, B = d["u_resample"].numel(), d["temperature"].numel()
    out_t = torch.full((R_t,), -9, dtype=torch.int32, device="cuda")
    out_n = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    rc = sv.lib().spec_verify_noalloc(
        _p(d["target_logits"]), _p(d["draft_logits"]), _p(toks), _p(d["u_accept"]),
        _p(d["u_resample"]), _p(d["temperature"]), B, _p(d["k_offsets"]), V, dtype,
        _p(out_t), _p(out_n), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, sv.lib().spec_last_error()
    return out_t, out_n


@pytest.mark.parametrize("case", [
    dict(B=48, k="ragged_1_10", V=32000, dtype="bf16", temperature="odd_greedy", seed=31),
    dict(B=20, k=[0, 1, 2, 3, 5, 8, 13, 21, 32, 4, 7, 1, 2, 2, 6, 9, 10, 3, 1, 1], V=16000,
         dtype="f32", temperature=0.9, seed=32),
    # a batch of the deferred epilogue (decisions and residual stream in one launch)
    dict(B=200, k="ragged_1_10", V=8192, dtype="bf16", temperature="odd_greedy", sigma_d=1.5, seed=34),
])
def test_noalloc_matches_spec_verify_twice(sv, case):
    w = workloads.make_case(**case)
    d = _device(w)
    toks = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"])
    ref_t, ref_n = sv.spec_verify(d["target_logits"], d["draft_logits"], toks, d["u_accept"],
                                  d["u_resample"], d["temperature"], d["k_offsets"])
    dt = sv.BF16 if w.dtype == "bf16" else sv.F32
    for _ in range(2):  # the second call finds the first call's leftovers in the array
        t, n = _noalloc_call(sv, d, toks, w.V, dt)
        torch.cuda.synchronize()
        assert torch.equal(t, ref_t) and torch.equal(n, ref_n)
    # the python wrapper marshals to the same entry point
    t2, n2 = sv.spec_verify_noalloc(d["target_logits"], d["draft_logits"], toks, d["u_accept"],
                                    d["u_resample"], d["temperature"], d["k_offsets"])
    torch.cuda.synchronize()
    assert torch.equal(t2, ref_t) and torch.equal(n2, ref_n)


def test_noalloc_refuses_batches_beyond_the_array(sv):
    limit = 48 << 20
    V = 262144  # bf16: a large vocabulary; B = 4096 needs far more scratch than the array
    assert sv.noalloc_bytes(4096, V, sv.BF16) > limit
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = sv.lib().spec_verify_noalloc(fake, fake, fake, fake, fake, fake, 4096, fake, V, sv.BF16,
                                      fake, fake, None)
    assert rc == -5  # SPEC_ERR_WORKSPACE
    assert b"scratch" in sv.lib().spec_last_error()
    assert sv.noalloc_bytes(512, 152064, sv.BF16) <= limit


def test_noalloc_wrapper_checks_its_inputs(sv):
    """The Python wrapper refuses what spec_verify refuses, before the C ABI
    sees a pointer: host tensors, mixed logit dtypes, non-contiguous views,
    a short k_offsets, and output buffers of the wrong type or size."""
    w = workloads.make_case(B=4, k=3, V=1000, dtype="f32", seed=33)
    d = _device(w)
    toks = sv.spec_draft_sample(d["draft_logits"], d["temperature"], d["u_draft"], d["k_offsets"])
    rest = (d["u_accept"], d["u_resample"], d["temperature"], d["k_offsets"])
    tl, dl = d["target_logits"], d["draft_logits"]
    with pytest.raises(ValueError):
        sv.spec_verify_noalloc(tl.cpu(), dl, toks, *rest)
    with pytest.raises(TypeError):
        sv.spec_verify_noalloc(tl, dl.to(torch.bfloat16), toks, *rest)
    strided = torch.empty((tl.shape[1], tl.shape[0]), dtype=tl.dtype, device="cuda").t()
    strided.copy_(tl)
    with pytest.raises(ValueError):
        sv.spec_verify_noalloc(strided, dl, toks, *rest)
    with pytest.raises(ValueError):
        sv.spec_verify_noalloc(tl, dl, toks, *rest[:3], d["k_offsets"][:-1])
    with pytest.raises(ValueError):
        sv.spec_verify_noalloc(tl, dl, toks, *rest, out_tokens=torch.empty(2, dtype=torch.int32, device="cuda"))
    with pytest.raises(TypeError):
        sv.spec_verify_noalloc(tl, dl, toks, *rest,
                               out_num_accepted=torch.empty(w.B, dtype=torch.int64, device="cuda"))
    # given buffers of the right kind are used as they are
    out_t = torch.empty(w.rows_target, dtype=torch.int32, device="cuda")
    out_n = torch.empty(w.B, dtype=torch.int32, device="cuda")
    t, n = sv.spec_verify_noalloc(tl, dl, toks, *rest, out_tokens=out_t, out_num_accepted=out_n)
    ref_t, ref_n = sv.spec_verify(tl, dl, toks, *rest)
    torch.cuda.synchronize()
    assert t is out_t and n is out_n
    assert torch.equal(t, ref_t) and torch.equal(n, ref_n)
