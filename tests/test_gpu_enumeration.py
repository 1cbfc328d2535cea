"""The losslessness check on the GPU (the tiny-vocabulary side check of the
B=8, V=32000 workload): the CUDA verify is evaluated at the midpoint of every
cell of its decision function on V = 8, with every drafted token x weighted
by q(x), and the law of each emitted slot must equal the target distribution
of its position: P_output(x) = min(q, p) + max(0, p - q) = p
(docs.ifdog.com "投机解码", section 无损保证：数学推导).

The cells and their weights come from the oracle pin's enumeration (cell
boundaries at alpha_i and at the cumulative masses C_v / Z, computed with
scipy in fp64); the GPU outputs are weighed with them.  The GPU decides in
fp32, so a cell narrower than its arithmetic error could fall on the other
side: the law must match p to 1e-6 plus the total weight of the cells whose
oracle margin is at most 1e-5 (where either decision is allowed), and the
tokens must equal the oracle's in every other cell."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from oracle_pins import emitted_law, enumerate_law, enumeration_rows, slot_of

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_61_gb300 as m
    m.lib()  # raises if the library is missing: no fallback
    return m


@pytest.mark.parametrize("k,seed,T", [(1, 1, 1.0), (2, 2, 1.0), (1, 3, 0.6), (2, 4, 0.6)])
def test_gpu_output_law_equals_p_over_enumeration_cells(sv, k, seed, T):
    V = 8
    t_rows, d_rows = enumeration_rows(k, seed, V)
    e = enumerate_law(oracle.load(), t_rows, d_rows, T)
    kw, w = e["kw"], e["weights"]
    B = len(kw["temperature"])
    assert B <= sv.MAX_B and abs(w.sum() - 1.0) < 1e-12
    d = {name: torch.from_numpy(np.ascontiguousarray(kw[name])).cuda()
         for name in ("target_logits", "draft_logits", "draft_tokens", "u_accept", "u_resample",
                      "temperature", "k_offsets")}
    gt, gn = sv.spec_verify(d["target_logits"], d["draft_logits"], d["draft_tokens"], d["u_accept"],
                            d["u_resample"], d["temperature"], d["k_offsets"])
    torch.cuda.synchronize()
    gt, gn = gt.cpu().numpy(), gn.cpu().numpy()
    assert (gn >= 0).all()
    slots = np.stack([gt[slot_of(kw["k_offsets"], b): slot_of(kw["k_offsets"], b) + k + 1] for b in range(B)])
    ok = e["margin"] > 1e-5
    slack = float(w[~ok].sum())
    for i in range(k + 1):
        np.testing.assert_allclose(emitted_law(w, slots, gn, i, V), e["p"][i], atol=1e-6 + slack, rtol=0,
                                   err_msg=f"GPU law of slot {i} != p_{i}")
    # outside flagged cells the GPU takes the oracle's decisions exactly
    assert ok.mean() > 0.8
    assert (gn[ok] == e["num"][ok]).all()
    assert (slots[ok] == e["slots"][ok]).all()
