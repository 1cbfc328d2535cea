"""Pins for the oracle's tree (multi-candidate) verify and tree drafting:
checks against what the mathematics fixes, independent of the oracle's code.
Each check takes an oracle library handle, so that the mutation tests can run
them against copies of the oracle with a planted mistake.

The tree rule is a reading (the pages draw candidate trees but give no
acceptance rule): children drawn i.i.d. from their parent's draft
distribution q are tried in index order; child j is accepted with
probability min(1, p^(j-1)(x)/q(x)), p^(0) = p, and each rejection replaces
p by norm(max(0, p - q)).  What pins it:
  * exact enumeration on tiny trees: the law of every emitted token equals
    the target distribution of the node it is drawn at (the single-candidate
    losslessness lemma of docs.ifdog.com '投机解码' 无损保证, applied once per
    candidate), for a root with three candidates (two levels of residual)
    and for a two-level tree;
  * a tree in which no node has two children is a chain: its outputs equal
    the chain oracle's, position by position;
  * greedy equals a brute-force walk with numpy.argmax (first occurrence),
    with duplicate sibling tokens;
  * tree drafting equals numpy.searchsorted on the parent's softmax;
  * data errors mark only their sequence; a bad node_offsets fails the call.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import softmax

import oracle


def sm(z, T):
    return softmax(np.asarray(z, dtype=np.float64) / T)


def _cells(probs):
    """[(lo, hi, v)]: the inverse-CDF cell of each token v of a distribution."""
    c = np.cumsum(probs) / probs.sum()
    out, lo = [], 0.0
    for v, hi in enumerate(c):
        if hi > lo:
            out.append((lo, float(hi), v))
        lo = max(lo, float(hi))
    return out


def _mid(lo, hi):
    m = np.float32((lo + hi) / 2)
    assert lo < float(m) < hi, "cell too narrow for an fp32 midpoint"
    return float(m)


def _resid(p, q):
    w = np.maximum(0.0, p - q)
    return w / w.sum() if w.sum() > 0 else p


def run_trees(lib, trees, T, V, dtype=np.float32):
    """trees: list of dicts with parent (local, -1 root), t_rows [n,V],
    d_rows [n,V], tokens [n], ua [n], ur [n].  One oracle call."""
    sizes = [len(t["parent"]) for t in trees]
    no = np.zeros(len(trees) + 1, dtype=np.int32)
    no[1:] = np.cumsum(sizes)
    par = np.concatenate([np.where(np.asarray(t["parent"]) >= 0, np.asarray(t["parent"]) + no[b], -1)
                          for b, t in enumerate(trees)]).astype(np.int32)
    cat = lambda key, dt: np.concatenate([np.asarray(t[key], dtype=dt) for t in trees])
    tl = np.concatenate([np.asarray(t["t_rows"], dtype=dtype).reshape(-1, V) for t in trees])
    dl = np.concatenate([np.asarray(t["d_rows"], dtype=dtype).reshape(-1, V) for t in trees])
    res = oracle.tree_verify(tl, dl, no, par, cat("tokens", np.int32), cat("ua", np.float32),
                             cat("ur", np.float32), np.full(len(trees), T, np.float32), lib=lib)
    return res, no


def enumerate_tree(lib, parent, t_rows, d_rows, T):
    """Exact law of the oracle's emitted tokens for one tree, with every
    child's token drawn from its parent's q and the uniforms uniform.  The
    walk below forms the cells of the reading (p, q from scipy); the oracle
    is evaluated at each cell's midpoint.  Returns a list of
    (weight, branch, emitted tokens, oracle tokens, num, last)."""
    n = len(parent)
    V = len(t_rows[0])
    p = [sm(r, T) for r in t_rows]
    q = [sm(r, T) for r in d_rows]
    children = [[c for c in range(n) if parent[c] == u] for u in range(n)]
    leaves = []

    def walk(tokens, weight, u, ua, ur, branch, emitted):
        # tokens: full assignment; walk the decisions from node u
        kids = children[u]
        if not kids:
            for lo, hi, v in _cells(p[u]):
                r = dict(ur)
                r[u] = _mid(lo, hi)
                leaves.append((weight * (hi - lo), branch + [("bonus", u)], emitted + [v], tokens, ua, r))
            return
        cur = p[u]
        for j, c in enumerate(kids):
            x = tokens[c]
            a = 1.0 if q[u][x] == 0 else min(1.0, cur[x] / q[u][x])
            if a > 0.0:
                a2 = dict(ua)
                a2[c] = _mid(0.0, a) if a < 1.0 else 0.5
                walk(tokens, weight * a, c, a2, ur, branch + [("acc", c)], emitted + [x])
            if a >= 1.0:
                return
            ua = dict(ua)
            ua[c] = _mid(a, 1.0)
            weight *= 1.0 - a
            branch = branch + [("rej", c)]
            cur = _resid(cur, q[u])
        for lo, hi, v in _cells(cur):
            r = dict(ur)
            r[u] = _mid(lo, hi)
            leaves.append((weight * (hi - lo), branch + [("draw", u)], emitted + [v], tokens, ua, r))

    # enumerate token assignments: each child from its parent's q
    for xs in np.ndindex(*([V] * (n - 1))):
        tokens = [0] + list(xs)
        wx = math.prod(q[parent[c]][tokens[c]] for c in range(1, n))
        if wx > 0.0:
            walk(tokens, wx, 0, {}, {}, [], [])

    trees = [dict(parent=parent, t_rows=t_rows, d_rows=d_rows, tokens=tk,
                  ua=[ua.get(i, 0.5) for i in range(n)], ur=[ur.get(i, 0.5) for i in range(n)])
             for _, _, _, tk, ua, ur in leaves]
    res, no = run_trees(lib, trees, T, V)
    assert res.rc == 0
    out = []
    for b, (w, br, em, _, _, _) in enumerate(leaves):
        g0 = int(no[b])
        out.append((w, br, em, res.tokens[g0:g0 + n], int(res.num_accepted[b]),
                    int(res.last_node[b]) - g0))
    return out, p


def check_tree_enumeration(lib, parent, seed, V, T):
    rng = np.random.default_rng(seed)
    n = len(parent)
    t_rows = (rng.standard_normal((n, V)) * 1.5).astype(np.float32)
    d_rows = (t_rows + rng.standard_normal((n, V)) * 0.8).astype(np.float32)
    leaves, p = enumerate_tree(lib, parent, t_rows, d_rows, T)
    W = sum(l[0] for l in leaves)
    assert abs(W - 1.0) < 1e-12, W
    for w, br, em, toks, num, last in leaves:
        # the oracle took the branch the reading takes at these uniforms
        assert num == len(em) - 1, (br, em, toks, num)
        assert list(toks[:len(em)]) == em, (br, em, toks)
        assert (toks[len(em):] == -1).all()
        end = br[-1][1]
        assert last == end, (br, last)
    # the first emitted token follows p at the root
    law = np.zeros(V)
    for w, br, em, *_ in leaves:
        law[em[0]] += w
    np.testing.assert_allclose(law, p[0], atol=1e-12, rtol=0, err_msg="first token law != p_root")
    # given that the walk moved to node c, the next emitted token follows p_c
    for c in range(1, n):
        mass, law = 0.0, np.zeros(V)
        for w, br, em, *_ in leaves:
            accs = [i for i, (kind, node) in enumerate(br) if kind == "acc"]
            pos = [k for k, i in enumerate(accs) if br[i][1] == c]
            if pos:
                mass += w
                law[em[pos[0] + 1]] += w
        if mass > 0:
            np.testing.assert_allclose(law / mass, p[c], atol=1e-11, rtol=0,
                                       err_msg=f"token after moving to node {c} != p_{c}")


def check_tree_chain_equivalence(lib):
    """A tree whose nodes have at most one child is the chain of the same
    rows: node i + 1 is drafted position i."""
    rng = np.random.default_rng(11)
    V = 24
    for T in (1.0, 0.7, 0.0):
        trees, seqs = [], []
        for b in range(30):
            k = int(rng.integers(0, 6))
            t_rows = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
            d_rows = (t_rows + rng.standard_normal((k + 1, V)) * 0.6).astype(np.float32)
            toks = [0] + [int(rng.integers(0, V)) for _ in range(k)]
            if T == 0 and k:
                # make some drafted tokens the target arg-max, so paths grow
                for i in range(1, k + 1):
                    if rng.random() < 0.7:
                        toks[i] = int(np.argmax(t_rows[i - 1]))
            ua = rng.random(k + 1).astype(np.float32)
            ur = rng.random(k + 1).astype(np.float32)
            trees.append(dict(parent=[-1] + list(range(k)), t_rows=t_rows, d_rows=d_rows, tokens=toks,
                              ua=ua, ur=ur))
            seqs.append((k, t_rows, d_rows[:k], toks[1:], ua[1:], ur))
        res, no = run_trees(lib, trees, T, V)
        ks = np.array([s[0] for s in seqs])
        ko = np.zeros(len(seqs) + 1, np.int32)
        ko[1:] = np.cumsum(ks)
        cres = oracle.verify(np.concatenate([s[1] for s in seqs]),
                             np.concatenate([s[2] for s in seqs]).reshape(-1, V),
                             np.concatenate([np.asarray(s[3], np.int32) for s in seqs]),
                             np.concatenate([s[4] for s in seqs]).astype(np.float32),
                             np.concatenate([s[5] for s in seqs]).astype(np.float32),
                             np.full(len(seqs), T, np.float32), ko, lib=lib)
        assert (res.num_accepted == cres.num_accepted).all(), (T, res.num_accepted, cres.num_accepted)
        for b, s in enumerate(seqs):
            k = s[0]
            assert (res.tokens[no[b]:no[b] + k + 1] == cres.tokens[ko[b] + b:ko[b] + b + k + 1]).all(), (T, b)


def check_tree_greedy_bruteforce(lib):
    """Greedy: the first child (in index order) whose token is the target
    arg-max; else the arg-max.  Sibling tokens repeat on purpose."""
    rng = np.random.default_rng(12)
    V = 6
    trees, want = [], []
    for b in range(40):
        n = int(rng.integers(1, 9))
        par = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        t_rows = rng.integers(-3, 3, size=(n, V)).astype(np.float32)  # ties likely
        toks = [0] + [int(rng.integers(0, 3)) for _ in range(1, n)]
        trees.append(dict(parent=par, t_rows=t_rows, d_rows=t_rows, tokens=toks,
                          ua=np.zeros(n), ur=np.zeros(n)))
        u, path = 0, []
        while True:
            am = int(np.argmax(t_rows[u]))
            nxt = [c for c in range(n) if par[c] == u and toks[c] == am]
            if not nxt:
                path.append(am)
                break
            path.append(toks[nxt[0]])
            u = nxt[0]
        want.append((path, u))
    res, no = run_trees(lib, trees, 0.0, V)
    for b, (path, last) in enumerate(want):
        n = len(trees[b]["parent"])
        got = res.tokens[no[b]:no[b] + n]
        assert res.num_accepted[b] == len(path) - 1, (b, res.num_accepted[b], path)
        assert list(got[:len(path)]) == path and (got[len(path):] == -1).all(), (b, got, path)
        assert res.last_node[b] - no[b] == last


def check_tree_draft_sample(lib):
    """Every non-root node draws from its parent's draft row: numpy's
    searchsorted of the cumulative softmax at u (strictly above u * total),
    arg-max at T = 0; roots give -1."""
    rng = np.random.default_rng(13)
    V = 16
    B = 12
    sizes = rng.integers(1, 7, size=B)
    no = np.zeros(B + 1, np.int32)
    no[1:] = np.cumsum(sizes)
    par = np.concatenate([[-1] + [int(no[b] + rng.integers(0, i)) for i in range(1, sizes[b])]
                          for b in range(B)]).astype(np.int32)
    N = int(no[-1])
    d = (rng.standard_normal((N, V)) * 2).astype(np.float32)
    T = np.where(np.arange(B) % 3 == 0, 0.0, 0.8).astype(np.float32)
    u = rng.random(N).astype(np.float32)
    res = oracle.tree_draft_sample(d, no, par, T, u, lib=lib)
    for b in range(B):
        for g in range(no[b], no[b + 1]):
            if par[g] < 0:
                assert res.tokens[g] == -1
                continue
            z = d[par[g]].astype(np.float64)
            if T[b] == 0:
                assert res.tokens[g] == int(np.argmax(z))
            else:
                pr = sm(z, float(T[b]))
                c = np.cumsum(pr)
                want = int(np.searchsorted(c, float(u[g]) * c[-1], side="right"))
                assert res.tokens[g] == min(want, V - 1), (g, res.tokens[g], want)


def check_tree_data_errors(lib):
    V = 8
    rng = np.random.default_rng(14)

    def tree(par, **kw):
        n = len(par)
        t = dict(parent=par, t_rows=rng.standard_normal((n, V)).astype(np.float32),
                 d_rows=rng.standard_normal((n, V)).astype(np.float32),
                 tokens=[0] + [1] * (n - 1), ua=np.full(n, 0.5), ur=np.full(n, 0.5))
        t.update(kw)
        return t

    good = tree([-1, 0, 0])
    bad_parent = tree([-1, 0, 2])                   # a node's parent is itself
    bad_token = tree([-1, 0], tokens=[0, V])        # token out of range
    nan_row = tree([-1, 0])
    nan_row["t_rows"][0, 3] = np.nan
    # strict test: p(x) = 0 with u = 0 rejects (u < alpha fails at alpha = 0)
    strict = tree([-1, 0], tokens=[0, 2], ua=[0.5, 0.0])
    strict["t_rows"][0, 2] = -np.inf
    res, no = run_trees(lib, [good, bad_parent, bad_token, nan_row, strict], 1.0, V)
    assert res.rc == 0
    assert res.num_accepted[0] >= 0
    assert list(res.num_accepted[1:4]) == [-1, -1, -1]
    assert (res.tokens[no[1]:no[4]] == -1).all()
    assert res.num_accepted[4] == 0 and res.tokens[no[4]] != 2
    # a node_offsets array with an empty sequence fails the whole call
    r = oracle.tree_verify(np.zeros((2, V), np.float32), np.zeros((2, V), np.float32),
                           np.array([0, 2, 2], np.int32), np.array([-1, 0], np.int32),
                           np.zeros(2, np.int32), np.zeros(2, np.float32), np.zeros(2, np.float32),
                           np.ones(2, np.float32), lib=lib)
    assert r.rc == -1 and (r.num_accepted == -1).all()


TREE_CHECKS = {
    "tree_enumeration_three_candidates": lambda lib: check_tree_enumeration(lib, [-1, 0, 0, 0], 21, 4, 1.0),
    "tree_enumeration_two_levels": lambda lib: check_tree_enumeration(lib, [-1, 0, 0, 1], 22, 4, 1.0),
    "tree_enumeration_two_levels_T0.6": lambda lib: check_tree_enumeration(lib, [-1, 0, 1, 0], 23, 4, 0.6),
    "tree_chain_equivalence": check_tree_chain_equivalence,
    "tree_greedy_bruteforce": check_tree_greedy_bruteforce,
    "tree_draft_sample": check_tree_draft_sample,
    "tree_data_errors": check_tree_data_errors,
}
