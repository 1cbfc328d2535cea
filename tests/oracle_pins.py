"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.  Each check takes an oracle library
handle so that the mutation tests can run the same checks against copies of
the oracle with a planted mistake.  Every check raises AssertionError on
failure.

What pins what:
  * softmax / log-sum-exp vs scipy.special (a library routine);
  * exact enumeration of the oracle's piecewise-constant decision function on
    a tiny vocabulary: the law of every emitted slot equals the target
    distribution p of that position (the losslessness theorem, docs.ifdog.com
    '投机解码' section 无损保证：数学推导; bbs.huaweicloud.com section 二.3), and
    the acceptance probability of position 0 equals 1 - Z with
    Z = sum max(0, p - q) (same section: Z is the rejection probability);
  * Z identity: sum max(0,p-q) = sum max(0,q-p) = 1 - sum min(p,q);
  * the resampled token always has p_v > q_v (residual support);
  * q = p accepts everything and the bonus equals the inverse-CDF draw of
    p_k computed with numpy.searchsorted;
  * greedy equals numpy.argmax (first occurrence on ties);
  * temperature: logits z at T equal logits z/T at T = 1 (T applies to every
    row);
  * hand-derived golden cases (tests/golden/hand_cases.json).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import logsumexp, softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cases.json")


def sm(z, T):
    return softmax(np.asarray(z, dtype=np.float64) / T)


def pack(seqs, dtype=np.float32):
    """seqs: list of dicts with t_rows [k+1,V], d_rows [k,V], tokens [k],
    u_accept [k], u_resample [k+1], T.  Returns oracle.verify kwargs."""
    ks = [len(s["tokens"]) for s in seqs]
    V = len(seqs[0]["t_rows"][0])
    k_offsets = np.zeros(len(seqs) + 1, dtype=np.int32)
    k_offsets[1:] = np.cumsum(ks)
    t = np.concatenate([np.asarray(s["t_rows"], dtype=dtype).reshape(-1, V) for s in seqs])
    d_list = [np.asarray(s["d_rows"], dtype=dtype).reshape(-1, V) for s in seqs]
    d = np.concatenate(d_list) if sum(ks) else np.zeros((0, V), dtype=dtype)
    cat = lambda key, dt: (np.concatenate([np.asarray(s[key], dtype=dt).ravel() for s in seqs])
                           if any(len(s[key]) for s in seqs) else np.zeros(0, dtype=dt))
    return dict(target_logits=t, draft_logits=d,
                draft_tokens=cat("tokens", np.int32),
                u_accept=cat("u_accept", np.float32),
                u_resample=cat("u_resample", np.float32),
                temperature=np.array([s["T"] for s in seqs], dtype=np.float32),
                k_offsets=k_offsets)


def slot_of(k_offsets, b):
    return int(k_offsets[b]) + b


# --------------------------------------------------------------------------
def check_softmax_vs_scipy(lib):
    rng = np.random.default_rng(7)
    for V in (1, 2, 5, 97, 1000):
        for T in (1.0, 0.7, 2.5):
            z = (rng.standard_normal(V) * 3).astype(np.float32)
            r = oracle.softmax_row(z, T, lib=lib)
            assert r is not None
            p, lse = r
            zz = z.astype(np.float64) / T
            assert abs(lse - logsumexp(zz)) <= 1e-12 * max(1.0, abs(lse))
            np.testing.assert_allclose(p, softmax(zz), rtol=1e-12, atol=1e-300)
    # bf16 bit patterns decode exactly
    z = (rng.standard_normal(64) * 4).astype(np.float32)
    import workloads
    bits = workloads.round_to_bf16_bits(z)
    vals = workloads.bf16_bits_to_f32(bits).astype(np.float64)
    p, lse = oracle.softmax_row(bits, 1.0, lib=lib)
    assert abs(lse - logsumexp(vals)) <= 1e-12 * max(1.0, abs(lse))


def _cells(breaks):
    """[(lo, hi, index)] for an increasing list of cumulative breakpoints
    (normalised to end at 1), skipping empty cells."""
    out = []
    lo = 0.0
    for v, hi in enumerate(breaks):
        if hi > lo:
            out.append((lo, hi, v))
        lo = max(lo, hi)
    return out


def _mid(lo, hi):
    m = np.float32((lo + hi) / 2)
    assert lo < float(m) < hi, "cell too narrow for an fp32 midpoint"
    return float(m)


def enumerate_law(lib, t_rows, d_rows, T):
    """Exact law of the oracle's outputs for one sequence with k = len(d_rows)
    drafted positions, with draft tokens drawn from q_i and uniforms uniform.
    Cells of (u_accept, u_resample) are formed from p, q computed here with
    scipy; the oracle is evaluated at each cell midpoint."""
    k = len(d_rows)
    V = len(t_rows[0])
    p = [sm(r, T) for r in t_rows]
    q = [sm(r, T) for r in d_rows]
    alpha = [np.minimum(1.0, np.where(qi > 0, pi / np.where(qi > 0, qi, 1), np.inf))
             for pi, qi in zip(p, q)]
    resid = []
    for i in range(k):
        w = np.maximum(0.0, p[i] - q[i])
        resid.append(np.cumsum(w) / w.sum())
    bonus = np.cumsum(p[k]) / p[k].sum()

    leaves, weights = [], []
    for xs in np.ndindex(*([V] * k)):
        wx = math.prod(q[i][xs[i]] for i in range(k))
        if wx == 0.0:
            continue

        def walk(i, ua, weight):
            if i == k:
                for lo, hi, v in _cells(bonus):
                    ur = [0.5] * (k + 1)
                    ur[k] = _mid(lo, hi)
                    leaves.append((xs, ua + [0.5] * (k - len(ua)), ur))
                    weights.append(weight * (hi - lo))
                return
            a = float(alpha[i][xs[i]])
            if a > 0.0:
                walk(i + 1, ua + [_mid(0.0, a) if a < 1.0 else 0.5], weight * a)
            if a < 1.0:
                for lo, hi, v in _cells(resid[i]):
                    ur = [0.5] * (k + 1)
                    ur[i] = _mid(lo, hi)
                    uu = ua + [_mid(a, 1.0)]
                    leaves.append((xs, uu + [0.5] * (k - len(uu)), ur))
                    weights.append(weight * (1.0 - a) * (hi - lo))

        walk(0, [], wx)

    seqs = [dict(t_rows=t_rows, d_rows=d_rows, tokens=list(xs), u_accept=ua,
                 u_resample=ur, T=T) for xs, ua, ur in leaves]
    kw = pack(seqs)
    res = oracle.verify(**kw, lib=lib)
    assert res.rc == 0
    weights = np.asarray(weights)
    B = len(seqs)
    slots = np.stack([res.tokens[slot_of(kw["k_offsets"], b): slot_of(kw["k_offsets"], b) + k + 1]
                      for b in range(B)])
    return dict(p=p, q=q, weights=weights, slots=slots, num=res.num_accepted, kw=kw, margin=res.margin)


def enumeration_rows(k, seed, V=8):
    """The tiny-vocabulary target and draft rows the enumeration pins use."""
    rng = np.random.default_rng(seed)
    t_rows = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    d_rows = (t_rows[:k] + rng.standard_normal((k, V)) * 0.8).astype(np.float32)
    return t_rows, d_rows


def emitted_law(weights, slots, num, i, V):
    """Law of output slot i over the enumeration cells (weighted), given that
    the slot holds a token (at least i drafted tokens accepted)."""
    emitted = num >= i
    mass = weights[emitted].sum()
    return np.array([weights[emitted & (slots[:, i] == y)].sum() for y in range(V)]) / mass


def check_enumeration(lib, k, seed, V=8, T=1.0):
    t_rows, d_rows = enumeration_rows(k, seed, V)
    e = enumerate_law(lib, t_rows, d_rows, T)
    w, slots, num, p, q = e["weights"], e["slots"], e["num"], e["p"], e["q"]
    assert abs(w.sum() - 1.0) < 1e-12
    assert (num >= 0).all()
    for i in range(k + 1):
        law = emitted_law(w, slots, num, i, V)  # slot i holds a token iff at least i accepted
        np.testing.assert_allclose(law, p[i], atol=1e-12, rtol=0,
                                   err_msg=f"law of slot {i} != p_{i}")
        # slots after the emitted one are -1
        assert (slots[num == i - 1, i:] == -1).all() if i > 0 else True
    # P(position 0 accepted) = sum_x min(p, q) = 1 - Z_0
    Z0 = np.maximum(0.0, p[0] - q[0]).sum()
    assert abs(w[num >= 1].sum() - (1.0 - Z0)) < 1e-12


def check_z_identity(lib):
    rng = np.random.default_rng(11)
    seqs, pq = [], []
    for V in (3, 17, 256, 5000):
        for s in range(3):
            t = (rng.standard_normal((2, V)) * 2).astype(np.float32)
            d = (t[:1] + rng.standard_normal((1, V))).astype(np.float32)
            p, q = sm(t[0], 1.0), sm(d[0], 1.0)
            cand = np.flatnonzero(p < q)
            x = int(cand[np.argmax(q[cand])])
            seqs.append(dict(t_rows=t, d_rows=d, tokens=[x], u_accept=[0.99999994],
                             u_resample=[0.5, 0.5], T=1.0))
            pq.append((p, q))
        # one vocabulary size per batch (rows share V)
        kw = pack(seqs)
        r = oracle.verify(**kw, lib=lib)
        for b, (p, q) in enumerate(pq):
            assert r.num_accepted[b] == 0
            Z = r.residual_mass[b]
            assert abs(Z - np.maximum(0.0, q - p).sum()) < 1e-12
            assert abs(Z - (1.0 - np.minimum(p, q).sum())) < 1e-12
            assert abs(Z - np.maximum(0.0, p - q).sum()) < 1e-12
            v = r.tokens[slot_of(kw["k_offsets"], b)]
            assert p[v] > q[v], "resampled token outside the residual support"
        seqs, pq = [], []


def check_q_equals_p_bonus(lib):
    rng = np.random.default_rng(5)
    V, k = 300, 4
    seqs, ps, us = [], [], []
    for s in range(20):
        t = (rng.standard_normal((k + 1, V)) * 2).astype(np.float32)
        ur = rng.random(k + 1).astype(np.float32)
        seqs.append(dict(t_rows=t, d_rows=t[:k].copy(), tokens=list(rng.integers(0, V, k)),
                         u_accept=rng.random(k).astype(np.float32), u_resample=ur, T=1.3))
        ps.append(sm(t[k], 1.3))
        us.append(float(ur[k]))
    kw = pack(seqs)
    r = oracle.verify(**kw, lib=lib)
    for b in range(len(seqs)):
        assert r.num_accepted[b] == k
        np.testing.assert_allclose(r.accept_prob[kw["k_offsets"][b]:kw["k_offsets"][b + 1]], 1.0,
                                   rtol=0, atol=1e-12)
        c = np.cumsum(ps[b])
        want = int(np.searchsorted(c, us[b] * c[-1], side="right"))
        assert r.tokens[slot_of(kw["k_offsets"], b) + k] == want


def check_greedy_bruteforce(lib):
    rng = np.random.default_rng(3)
    V, k = 12, 5
    seqs, want = [], []
    for s in range(200):
        t = rng.integers(-3, 4, size=(k + 1, V)).astype(np.float32)  # many ties
        am = np.argmax(t, axis=1)
        x = [int(am[i]) if rng.random() < 0.7 else int(rng.integers(0, V)) for i in range(k)]
        seqs.append(dict(t_rows=t, d_rows=np.zeros((k, V), np.float32), tokens=x,
                         u_accept=[0.5] * k, u_resample=[0.5] * (k + 1), T=0.0))
        n = next((i for i in range(k) if x[i] != am[i]), k)
        want.append((n, x[:n] + [int(am[n])] + [-1] * (k - n)))
    kw = pack(seqs)
    r = oracle.verify(**kw, lib=lib)
    for b, (n, toks) in enumerate(want):
        o = slot_of(kw["k_offsets"], b)
        assert r.num_accepted[b] == n
        assert list(r.tokens[o:o + k + 1]) == toks


def check_temperature_equivalence(lib):
    rng = np.random.default_rng(9)
    V, k = 64, 3
    base = []
    for s in range(30):
        t = (rng.standard_normal((k + 1, V))).astype(np.float32)
        d = (t[:k] + rng.standard_normal((k, V)) * 0.7).astype(np.float32)
        base.append(dict(t_rows=t, d_rows=d, tokens=list(rng.integers(0, V, k)),
                         u_accept=rng.random(k).astype(np.float32),
                         u_resample=rng.random(k + 1).astype(np.float32)))
    a = pack([dict(s, T=0.5) for s in base])
    bb = pack([dict(s, t_rows=2 * s["t_rows"], d_rows=2 * s["d_rows"], T=1.0) for s in base])
    ra = oracle.verify(**a, lib=lib)
    rb = oracle.verify(**bb, lib=lib)
    assert (ra.tokens == rb.tokens).all() and (ra.num_accepted == rb.num_accepted).all()
    np.testing.assert_array_equal(ra.accept_prob, rb.accept_prob)


def _golden_logits(case, key_probs, key_logits):
    if key_logits in case:
        return np.asarray(case[key_logits], dtype=np.float32)
    P = np.asarray(case[key_probs], dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(P).astype(np.float32)


def check_golden(lib):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        t = _golden_logits(c, "target_probs", "target_logits")
        V = t.shape[1]
        d = (_golden_logits(c, "draft_probs", "draft_logits") if c.get("draft_tokens")
             else np.zeros((0, V), np.float32))
        seq = dict(t_rows=t, d_rows=d, tokens=c["draft_tokens"], u_accept=c["u_accept"],
                   u_resample=c["u_resample"], T=c["temperature"])
        kw = pack([seq])
        r = oracle.verify(**kw, lib=lib)
        assert list(r.tokens) == c["expect_tokens"], c["name"]
        assert r.num_accepted[0] == c["expect_num_accepted"], c["name"]
        if c.get("expect_alpha") is not None:
            np.testing.assert_allclose(r.accept_prob, c["expect_alpha"], rtol=0,
                                       atol=c.get("alpha_tol", 1e-6), err_msg=c["name"])
        if "expect_residual_mass" in c:
            # logits are fp32-rounded logarithms: values agree to ~1e-7
            assert abs(r.residual_mass[0] - c["expect_residual_mass"]) < 1e-6, c["name"]


ALL_CHECKS = {
    "softmax_vs_scipy": check_softmax_vs_scipy,
    "enumeration_k1": lambda lib: check_enumeration(lib, 1, seed=1),
    "enumeration_k2": lambda lib: check_enumeration(lib, 2, seed=2),
    "enumeration_k2_T0.6": lambda lib: check_enumeration(lib, 2, seed=4, T=0.6),
    "z_identity": check_z_identity,
    "q_equals_p_bonus": check_q_equals_p_bonus,
    "greedy_bruteforce": check_greedy_bruteforce,
    "temperature_equivalence": check_temperature_equivalence,
    "golden": check_golden,
}
