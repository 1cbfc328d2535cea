"""GPU parity at the sizes the C ABI declares as its limits: the largest
vocabulary (MAX_V = 2^24 columns: 2048 chunks and 16384 sub-chunk partials
per row) and the most sequences per call (MAX_B = 4096, with k_b spanning
0..MAX_K).  The outputs are checked against the fp64 oracle under the usual
parity rules, and the fused round and the host-buffer round must equal the
separate calls bit for bit."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import workloads
from parity import gpu_draft_sample, gpu_verify, run_and_compare, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_61_gb300 as m
    m.lib()  # raises if the library is missing: no fallback
    return m


def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the same values as fp32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.fixture(scope="module")
def largest_vocabulary():
    # two sequences, k = 1 and 2: 5 target and 3 draft rows of 2^24 columns
    return workloads.make_case(B=2, k=[1, 2], V=1 << 24, dtype="bf16", temperature=1.0, seed=321,
                               name="B2_k1,2_V16777216_bf16")


def round_equals_separate_calls(sv, d):
    toks = gpu_draft_sample(d)
    t0, n0 = gpu_verify(d, toks, aux=False)
    args = (d["u_accept"], d["u_resample"], d["temperature"], d["k_offsets"])
    toks2, t2, n2 = sv.spec_round(d["target_logits"], d["draft_logits"], d["u_draft"], *args)
    torch.cuda.synchronize()
    assert torch.equal(toks2, toks) and torch.equal(t2, t0) and torch.equal(n2, n0)
    return toks, t0, n0


def test_largest_vocabulary_bf16(sv, largest_vocabulary):
    w = largest_vocabulary
    assert w.V == sv.MAX_V
    rep = run_and_compare(w)
    assert rep["sequences"] == 2
    round_equals_separate_calls(sv, to_device(w))


def test_largest_vocabulary_f32(sv, largest_vocabulary):
    w = dataclasses.replace(largest_vocabulary, dtype=workloads.F32,
                            target_logits=widen(largest_vocabulary.target_logits),
                            draft_logits=widen(largest_vocabulary.draft_logits),
                            name="B2_k1,2_V16777216_f32")
    run_and_compare(w)
    round_equals_separate_calls(sv, to_device(w))


def test_fixed_scratch_at_the_largest_vocabulary(sv, largest_vocabulary):
    """The allocation-free entry point at V = 2^24: two sequences fit its
    fixed scratch and give spec_verify's outputs bit for bit; six do not
    (the scratch grows with B) and are refused with SPEC_ERR_WORKSPACE
    before anything runs."""
    w = largest_vocabulary
    d = to_device(w)
    toks = gpu_draft_sample(d)
    t0, n0 = gpu_verify(d, toks, aux=False)
    t1, n1 = sv.spec_verify_noalloc(d["target_logits"], d["draft_logits"], toks, d["u_accept"],
                                    d["u_resample"], d["temperature"], d["k_offsets"])
    torch.cuda.synchronize()
    assert torch.equal(t1, t0) and torch.equal(n1, n0)

    B = 6
    assert sv.noalloc_bytes(w.B, w.V, sv.BF16) <= sv.NOALLOC_SCRATCH_BYTES < sv.noalloc_bytes(B, w.V, sv.BF16)
    # k_b = 1: two target rows and one draft row per sequence
    tl = torch.zeros((2 * B, w.V), dtype=torch.bfloat16, device="cuda")
    dl = torch.zeros((B, w.V), dtype=torch.bfloat16, device="cuda")
    half = torch.full((2 * B,), 0.5, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_noalloc(tl, dl, torch.zeros(B, dtype=torch.int32, device="cuda"), half[:B], half,
                               torch.ones(B, device="cuda"), torch.arange(B + 1, dtype=torch.int32, device="cuda"))
    assert e.value.code == -5


def test_most_sequences(sv):
    """B = MAX_B with every k from 0 to MAX_K present, a 264-column
    vocabulary (one ragged 2 KB sub-chunk per row), greedy and sampled
    sequences alternating."""
    ks = np.random.default_rng(5).integers(0, sv.MAX_K + 1, sv.MAX_B)
    ks[:sv.MAX_K + 1] = np.arange(sv.MAX_K + 1)
    w = workloads.make_case(B=sv.MAX_B, k=list(ks), V=264, dtype="bf16", temperature="odd_greedy", seed=322,
                            name="B4096_k0to32_V264_bf16")
    rep = run_and_compare(w)
    assert rep["sequences"] == sv.MAX_B
    d = to_device(w)
    toks, t0, n0 = round_equals_separate_calls(sv, d)

    def h(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(torch.bfloat16) if a.dtype == np.uint16 else x).pin_memory()

    hd, ht, hn = sv.spec_round_host(h(w.target_logits), h(w.draft_logits), h(w.u_draft), h(w.u_accept),
                                    h(w.u_resample), h(w.temperature), h(w.k_offsets))
    assert torch.equal(hd, toks.cpu()) and torch.equal(ht, t0.cpu()) and torch.equal(hn, n0.cpu())
