"""Pins of the oracle's best-first heap with parent-conditioned edge scores and
of its edge-term tables (CPU only).

- heap_select without edge terms is the DDTree heap (pinned by brute force);
- with non-positive edge scores it returns the B best prefixes of the whole
  lattice, found here by enumerating every prefix;
- with edge scores of either sign it keeps the best-first invariant: a node
  is never popped while a better one waits in the frontier;
- with the normalised Markov correction and no width limit it selects what
  DARTree's depth-wise supertree + Top-B selects ([DARTree] Lemma 1);
- the TDES table matches a hand-computed two-unit scorer, its ReLU cut, and a
  float64 restatement within rounding."""
import itertools

import numpy as np
import pytest

import oracle


def _lattice(L, V, K, seed, scale=1.5, quant=False):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((L, V)) * scale).astype(np.float32)
    if quant:  # coarse values: many equal logits, hence equal scores
        x = np.round(x * 2) / 2
    _, _, ids, lps = oracle.candidates(x, K)
    return x, ids, lps


def _same(a, b):
    assert a.n == b.n, (a.n, b.n)
    n = a.n
    for f in ("tok", "parent", "depth", "rank"):
        assert np.array_equal(getattr(a, f)[:n], getattr(b, f)[:n]), f
    assert np.array_equal(a.score[:n], b.score[:n])


@pytest.mark.parametrize("quant", [False, True])
def test_heap_without_edge_terms_is_ddtree(quant):
    for seed in range(12):
        L, V, K = 4, 30, 5
        _, ids, lps = _lattice(L, V, K, seed, quant=quant)
        for B in (1, 7, 40, 1000):
            _same(oracle.heap_select(lps, ids, B), oracle.ddtree(lps, ids, B))


def _edge_t(lps, E, d, i, j):
    """fp32 edge score of candidate j of position d (1-based) under parent row i."""
    return np.float32(lps[d - 1, j]) + np.float32(E[d - 1, i, j])


def _orders(lps, E):
    """Order position of every child under every parent row: (t desc, j asc)."""
    L, K = lps.shape
    pos = np.zeros((L, K, K), np.int64)
    for d in range(1, L + 1):
        for i in range(K):
            t = [_edge_t(lps, E, d, i, j) for j in range(K)]
            order = sorted(range(K), key=lambda j: (-t[j], j))
            for p, j in enumerate(order):
                pos[d - 1, i, j] = p
    return pos


def _enumerate(lps, E):
    """Every prefix of the lattice: (score, order descriptor, rank path)."""
    L, K = lps.shape
    pos = _orders(lps, E)
    out = []
    for d in range(1, L + 1):
        for path in itertools.product(range(K), repeat=d):
            s = np.float32(0.0)
            desc = []
            prev = 0
            for k, c in enumerate(path):
                s = np.float32(s + _edge_t(lps, E, k + 1, prev, c))
                desc.append(int(pos[k, prev, c]))
                prev = c
            out.append((float(s), tuple(desc), path))
    return out


def _rank_paths(t):
    paths = []
    for n in range(1, t.n):
        p, a = [], n
        while a != 0:
            p.append(int(t.rank[a]))
            a = int(t.parent[a])
        paths.append(tuple(reversed(p)))
    return paths


def test_heap_is_the_best_prefixes_when_edges_do_not_raise_scores():
    for seed in range(6):
        L, V, K = 3, 12, 3
        _, ids, lps = _lattice(L, V, K, seed)
        rng = np.random.default_rng(100 + seed)
        E = -np.abs(rng.standard_normal((L, K, K))).astype(np.float32)  # t = lp + E <= 0
        allp = sorted(_enumerate(lps, E), key=lambda e: (-e[0], e[1]))
        for B in range(1, len(allp) + 2):
            t = oracle.heap_select(lps, ids, B, E=E)
            want = allp[:B]
            assert _rank_paths(t) == [e[2] for e in want], (seed, B)
            assert np.array_equal(t.score[1:t.n], np.array([e[0] for e in want], np.float32))


def test_heap_best_first_invariant_with_edges_of_either_sign():
    for seed in range(10):
        L, V, K = 4, 16, 4
        _, ids, lps = _lattice(L, V, K, seed)
        rng = np.random.default_rng(200 + seed)
        E = (rng.standard_normal((L, K, K)) * 3).astype(np.float32)  # some children outscore parents
        pos = _orders(lps, E)
        for B in (5, 30, 200):
            t = oracle.heap_select(lps, ids, B, E=E)
            n = t.n
            assert n - 1 == min(B, sum(K ** d for d in range(1, L + 1)))
            desc, key = {0: ()}, {}
            prow = {0: 0}
            for v in range(1, n):
                p = int(t.parent[v])
                assert 0 <= p < v and t.depth[v] == t.depth[p] + 1  # parents first
                c = int(t.rank[v])
                assert t.tok[v] == ids[t.depth[v] - 1, c]
                assert t.score[v] == np.float32(t.score[p] + _edge_t(lps, E, int(t.depth[v]), prow[p], c))
                desc[v] = desc[p] + (int(pos[t.depth[v] - 1, prow[p], c]),)
                prow[v] = c
                key[v] = (-float(t.score[v]), desc[v])
            # pred(v): previous sibling in the parent's order, else the parent
            where = {(int(t.parent[v]), desc[v][-1]): v for v in range(1, n)}
            for v in range(1, n):
                pr = int(t.parent[v]) if desc[v][-1] == 0 else where[(int(t.parent[v]), desc[v][-1] - 1)]
                assert pr < v
                # every node popped after v whose predecessor was popped before v
                # was already waiting when v was popped, so it cannot be better
                for k in range(v + 1, n):
                    pk = int(t.parent[k]) if desc[k][-1] == 0 else where[(int(t.parent[k]), desc[k][-1] - 1)]
                    if pk < v:
                        assert key[v] < key[k], (seed, B, v, k)


def test_heap_with_normalised_markov_term_equals_dartree_without_width_limit():
    L, V, K, R = 3, 40, 3, 4
    for seed in range(5):
        x, ids, lps = _lattice(L, V, K, seed)
        rng = np.random.default_rng(300 + seed)
        U = (rng.standard_normal((V, R)) * 0.5).astype(np.float32)
        Vt = (rng.standard_normal((V, R)) * 0.5).astype(np.float32)
        root = int(rng.integers(V))
        z = oracle.markov_norm(x, ids, U, Vt, root)
        E = oracle.markov_table(ids, U, Vt, root)
        for B in (4, 11, 39):
            d, info, _ = oracle.dartree(lps, ids, U, Vt, root, K ** (L - 1) * K, 0.0, B, znorm=z)
            assert info["violations"] == 0 and info["topb_equals_bestfirst"]
            h = oracle.heap_select(lps, ids, B, E=E, znorm=z)
            assert _rank_paths(h) == _rank_paths(d), (seed, B)
            assert np.array_equal(h.score[:h.n], d.score[:d.n])


def test_markov_table_rows():
    L, V, K, R = 3, 25, 4, 6
    _, ids, _ = _lattice(L, V, K, 1)
    rng = np.random.default_rng(4)
    U = rng.standard_normal((V, R)).astype(np.float32)
    Vt = rng.standard_normal((V, R)).astype(np.float32)
    E = oracle.markov_table(ids, U, Vt, 7)
    assert np.allclose(E[0, 0], U[7].astype(np.float64) @ Vt[ids[0]].T.astype(np.float64), atol=1e-5)
    assert np.all(E[0, 1:] == 0)
    for d in range(1, L):
        ref = U[ids[d - 1]].astype(np.float64) @ Vt[ids[d]].T.astype(np.float64)
        assert np.allclose(E[d], ref, atol=1e-5)
    assert np.all(oracle.markov_table(ids, U, Vt, -1)[0] == 0)


# ---------------------------------------------------------------------------
# TDES edge scorer
# ---------------------------------------------------------------------------
def test_tdes_two_unit_scorer_by_hand():
    # Two hidden units.  Tokens: 0, 1, 2.  Positions 1 and 2 have candidates
    # [0, 1] and [2, 0]; the root token is 1.
    #   Ap[1] = (0.5, -1), Ac[0] = (0.25, 2), Dd[0] = (0.25, -0.5), w = (2, -1),
    #   b0 = 0.5, s = 0.75:
    #   edge root(1) -> 0 at depth 1: a = (0.5+0.25+0.25, -1+2-0.5) = (1, 0.5),
    #   f = 2*1 - 1*0.5 + 0.5 = 2, E = 0.75 * 2 = 1.5.
    #   Ac[1] = (-2, 0): a = (0.5-2+0.25, -1+0-0.5) = (-1.25, -1.5): both cut,
    #   f = b0 = 0.5, E = 0.375.
    #   edge 0 -> 2 at depth 2 with Ap[0] = (1, 1), Ac[2] = (-0.5, 0.25),
    #   Dd[1] = (0, 0.5): a = (0.5, 1.75), f = 2*0.5 - 1.75 + 0.5 = -0.25,
    #   E = -0.1875.
    Ap = np.array([[1, 1], [0.5, -1], [0, 0]], np.float32)
    Ac = np.array([[0.25, 2], [-2, 0], [-0.5, 0.25]], np.float32)
    Dd = np.array([[0.25, -0.5], [0, 0.5]], np.float32)
    w = np.array([2, -1], np.float32)
    ids = np.array([[0, 1], [2, 0]], np.int32)
    E = oracle.tdes_table(ids, Ap, Ac, Dd, w, 0.5, 0.75, 1)
    assert E[0, 0, 0] == 1.5 and E[0, 0, 1] == 0.375 and np.all(E[0, 1] == 0)
    assert E[1, 0, 0] == -0.1875


def test_tdes_relu_cut_and_scale():
    L, V, K, H = 3, 20, 4, 8
    _, ids, _ = _lattice(L, V, K, 2)
    rng = np.random.default_rng(5)
    Ap = rng.standard_normal((V, H)).astype(np.float32)
    Ac = rng.standard_normal((V, H)).astype(np.float32)
    w = rng.standard_normal(H).astype(np.float32)
    Dd = np.full((L, H), -100.0, np.float32)  # every hidden unit cut: f = b0
    E = oracle.tdes_table(ids, Ap, Ac, Dd, w, 0.25, 2.0, 3)
    assert np.all(E[0, 0] == 0.5) and np.all(E[1:] == 0.5) and np.all(E[0, 1:] == 0)
    assert np.all(oracle.tdes_table(ids, Ap, Ac, Dd, w, 0.25, 2.0, -1)[0] == 0)  # no root token: no term


def test_tdes_matches_float64_restatement():
    L, V, K, H = 4, 50, 5, 32
    _, ids, _ = _lattice(L, V, K, 3)
    rng = np.random.default_rng(6)
    Ap = rng.standard_normal((V, H)).astype(np.float32)
    Ac = rng.standard_normal((V, H)).astype(np.float32)
    Dd = rng.standard_normal((L, H)).astype(np.float32)
    w = (rng.standard_normal(H) * 0.3).astype(np.float32)
    b0, s, root = -0.2, 1.3, 11
    E = oracle.tdes_table(ids, Ap, Ac, Dd, w, b0, s, root)

    def f(p, c, d):
        a = Ap[p].astype(np.float64) + Ac[c] + Dd[d - 1]
        return s * (float(np.maximum(a, 0) @ w.astype(np.float64)) + b0)

    for j in range(K):
        assert abs(E[0, 0, j] - f(root, ids[0, j], 1)) < 1e-4
    for d in range(2, L + 1):
        for i in range(K):
            for j in range(K):
                assert abs(E[d - 1, i, j] - f(ids[d - 2, i], ids[d - 1, j], d)) < 1e-4
