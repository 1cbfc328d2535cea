"""CPU tests of the fp64 oracle against its pins (no GPU)."""
from __future__ import annotations

import numpy as np
import pytest
from scipy.stats import chisquare

import oracle
import workloads
from oracle_pins import ALL_CHECKS, pack, slot_of, sm


@pytest.mark.parametrize("name", sorted(ALL_CHECKS))
def test_pin(name, oracle_lib):
    ALL_CHECKS[name](oracle_lib)


def _pool(counts, expect, min_expect=5.0):
    """Pool the cells with small expected counts into one (chi-square
    validity); the pooled cell is dropped if it expects nothing."""
    keep = expect > min_expect
    c, e = counts[keep].astype(np.float64), expect[keep]
    if expect[~keep].sum() > 0:
        c = np.append(c, counts[~keep].sum())
        e = np.append(e, expect[~keep].sum())
    return c, e * (c.sum() / e.sum())


def _shared_pq_batch(N, V, k, T, seed):
    """N sequences sharing one set of rows; draft tokens drawn from q by the
    oracle's own draft sampler with independent uniforms."""
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((k + 1, V)) * 1.5 - np.log1p(np.arange(V)) * 0.5).astype(np.float32)
    d = (t[:k] + rng.standard_normal((k, V)) * 0.6).astype(np.float32)
    k_offsets = np.arange(N + 1, dtype=np.int32) * k
    temp = np.full(N, T, np.float32)
    dl = np.tile(d, (N, 1))
    tl = np.tile(t, (N, 1))
    u = workloads.uniforms(np.random.Generator(np.random.Philox(seed)), N * k * 2 + N * (k + 1))
    u_draft, u_accept, u_res = u[:N * k], u[N * k:2 * N * k], u[2 * N * k:]
    ds = oracle.draft_sample(dl, temp, u_draft, k_offsets)
    assert ds.rc == 0 and (ds.tokens >= 0).all()
    r = oracle.verify(tl, dl, ds.tokens, u_accept, u_res, temp, k_offsets, nthreads=4)
    return t, d, ds, r, k_offsets


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_chi_square_emitted_tokens(T):
    """The first emitted token of every sequence, and the second one of the
    sequences that accepted position 0, follow p_0 and p_1 (the pages'
    losslessness claim), by a chi-square test with fixed seeds."""
    N, V, k = 1 << 15, 40, 2
    t, d, ds, r, ko = _shared_pq_batch(N, V, k, T, seed=17 if T == 1.0 else 18)
    slots = r.tokens.reshape(N, k + 1)
    for i in range(2):
        sel = r.num_accepted >= i
        counts = np.bincount(slots[sel, i], minlength=V)
        expect = sm(t[i], T) * sel.sum()
        stat, pval = chisquare(*_pool(counts, expect))
        assert pval > 1e-4, (i, pval)
    # acceptance rate of position 0 ~ 1 - Z_0
    p0, q0 = sm(t[0], T), sm(d[0], T)
    Z0 = np.maximum(0, p0 - q0).sum()
    acc = (r.num_accepted >= 1).mean()
    assert abs(acc - (1 - Z0)) < 5 * np.sqrt(Z0 * (1 - Z0) / N)


def test_draft_sample_distribution():
    """Draft sampling draws from softmax(z/T): chi-square of many draws from
    one row, plus argmax for T = 0."""
    rng = np.random.default_rng(21)
    V, N = 30, 1 << 14
    z = (rng.standard_normal(V) * 1.2).astype(np.float32)
    dl = np.tile(z, (N, 1))
    ko = np.arange(N + 1, dtype=np.int32)
    u = workloads.uniforms(np.random.Generator(np.random.Philox(3)), N)
    r = oracle.draft_sample(dl, np.full(N, 0.8, np.float32), u, ko)
    counts = np.bincount(r.tokens, minlength=V)
    e = sm(z, 0.8) * N
    _, pval = chisquare(*_pool(counts, e))
    assert pval > 1e-4
    g = oracle.draft_sample(dl[:4], np.zeros(4, np.float32), u[:4], ko[:5])
    assert (g.tokens == np.argmax(z)).all()
    # u in normalised CDF units: the draw is the searchsorted position
    c = np.cumsum(sm(z, 0.8))
    want = np.searchsorted(c, u.astype(np.float64) * c[-1], side="right")
    assert (r.tokens == want).all()


def test_unused_uniforms_do_not_matter():
    w = workloads.make_case(B=16, k=6, V=500, seed=5)
    ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
    r0 = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample,
                       w.temperature, w.k_offsets)
    ua, ur = w.u_accept.copy(), w.u_resample.copy()
    rng = np.random.default_rng(0)
    for b in range(w.B):
        n = r0.num_accepted[b]
        k0, k = int(w.k_offsets[b]), int(w.k[b])
        ua[k0 + n + 1:k0 + k] = rng.random(max(0, k - n - 1)).astype(np.float32)
        o = k0 + b
        for j in range(k + 1):
            if j != n:
                ur[o + j] = np.float32(rng.random())
    r1 = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, ua, ur, w.temperature,
                       w.k_offsets)
    assert (r0.tokens == r1.tokens).all() and (r0.num_accepted == r1.num_accepted).all()


def test_invalid_inputs_mark_only_their_sequence():
    w = workloads.make_case(B=6, k=3, V=100, seed=8)
    tl, dl = w.target_logits.copy(), w.draft_logits.copy()
    toks = np.zeros(w.rows_draft, np.int32)
    temp = w.temperature.copy()
    tl[1 * 4 + 2, 7] = np.nan          # seq 1: NaN in a target row
    dl[2 * 3 + 0, 3] = np.inf          # seq 2: +inf in a draft row
    toks[3 * 3 + 1] = 100              # seq 3: token out of range
    temp[4] = -1.0                     # seq 4: bad temperature
    tl[5 * 4 + 3, :] = -np.inf         # seq 5: bonus row entirely -inf
    r = oracle.verify(tl, dl, toks, w.u_accept, w.u_resample, temp, w.k_offsets)
    assert r.num_accepted[0] >= 0
    for b in range(1, 6):
        assert r.num_accepted[b] == -1
        o = slot_of(w.k_offsets, b)
        assert (r.tokens[o:o + 4] == -1).all()
    # invalid offsets: the whole call is rejected
    bad = w.k_offsets.copy()
    bad[2] = bad[1] - 1
    r = oracle.verify(tl, dl, toks, w.u_accept, w.u_resample, temp, bad)
    assert r.rc == -1 and (r.num_accepted == -1).all()
    big = np.array([0, 33], np.int32)
    r = oracle.verify(np.zeros((34, 4), np.float32), np.zeros((33, 4), np.float32),
                      np.zeros(33, np.int32), np.zeros(33, np.float32),
                      np.zeros(34, np.float32), np.ones(1, np.float32), big)
    assert r.rc == -1


def test_greedy_nan_row_is_error():
    kw = pack([dict(t_rows=np.array([[0, 1, np.nan], [1, 0, 0]], np.float32),
                    d_rows=np.zeros((1, 3), np.float32), tokens=[1], u_accept=[0.5],
                    u_resample=[0.5, 0.5], T=0.0)])
    r = oracle.verify(**kw)
    assert r.num_accepted[0] == -1 and (r.tokens == -1).all()


def test_bf16_and_f32_agree_on_same_values():
    """bf16 inputs are decoded exactly: feeding the decoded values as fp32
    gives identical decisions."""
    w = workloads.make_case(B=8, k=4, V=300, dtype=workloads.BF16, seed=12)
    ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
    a = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample,
                      w.temperature, w.k_offsets)
    tf = workloads.bf16_bits_to_f32(w.target_logits)
    df = workloads.bf16_bits_to_f32(w.draft_logits)
    b = oracle.verify(tf, df, ds.tokens, w.u_accept, w.u_resample, w.temperature, w.k_offsets)
    assert (a.tokens == b.tokens).all()
    np.testing.assert_array_equal(a.accept_prob, b.accept_prob)


def test_threads_do_not_change_results():
    w = workloads.make_case(B=24, k="ragged_1_10", V=700, seed=4, temperature="odd_greedy")
    ds = oracle.draft_sample(w.draft_logits, w.temperature, w.u_draft, w.k_offsets)
    a = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample,
                      w.temperature, w.k_offsets, nthreads=1)
    b = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample,
                      w.temperature, w.k_offsets, nthreads=4)
    assert (a.tokens == b.tokens).all()
    sub = oracle.verify(w.target_logits, w.draft_logits, ds.tokens, w.u_accept, w.u_resample,
                        w.temperature, w.k_offsets, seq_list=[3, 7, 20])
    for bb in (3, 7, 20):
        o = slot_of(w.k_offsets, bb)
        kk = int(w.k[bb])
        assert (sub.tokens[o:o + kk + 1] == a.tokens[o:o + kk + 1]).all()


def test_generator_is_deterministic_and_shaped():
    a = workloads.make_config(1)
    b = workloads.make_config(1)
    assert np.array_equal(a.target_logits, b.target_logits)
    assert a.target_logits.shape == (20, 1000) and a.draft_logits.shape == (16, 1000)
    assert a.u_resample.shape == (20,) and a.u_accept.shape == (16,)
    u = np.concatenate([a.u_accept, a.u_resample, a.u_draft]).astype(np.float64)
    assert ((u * (1 << 24)) == np.floor(u * (1 << 24))).all() and (u < 1).all()
    c = workloads.make_case(B=10, k="ragged_1_10", V=64, temperature="odd_greedy",
                            sigma_d="uniform_0.2_1.5", dtype=workloads.BF16)
    assert c.target_logits.dtype == np.uint16 and c.rows_target == c.rows_draft + 10
    assert (c.temperature[1::2] == 0).all() and (c.temperature[::2] == 1).all()
    assert c.k.min() >= 1 and c.k.max() <= 10


def test_generator_row_arrangements():
    """Without noise a target row is the Zipf ranks -a ln(1 + pi_r(v)) laid out
    by its permutation pi_r.  The default draws one arrangement per workload
    and rotates it per row (every row is a cyclic shift of the first);
    perm="per_row" draws an independent permutation for every row (no row is
    a cyclic shift of another)."""
    kw = dict(B=3, k=2, V=48, sigma_t=0.0, sigma_d=0.0, seed=5)
    base = np.sort((-1.1 * np.log1p(np.arange(48, dtype=np.float64))).astype(np.float32))
    for perm, cyclic in (("rotated", True), ("per_row", False)):
        w = workloads.make_case(perm=perm, **kw)
        rows = w.target_logits
        for r in rows:  # every row holds each Zipf rank exactly once
            assert np.array_equal(np.sort(r), base)
        shifts = [any(np.array_equal(rows[i], np.roll(rows[0], c)) for c in range(48))
                  for i in range(1, len(rows))]
        assert all(shifts) if cyclic else not any(shifts), perm
