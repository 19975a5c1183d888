"""Pins of the oracle's two further T=1 walks (CPU only).

- one residual per rejected sibling (oracle.verify_t1(..., rule="iter_residual")):
  child c_1 against p, child c_i against r_{i-1} = [r_{i-2} - q]_+ normalised,
  the replacement from the residual left by all rejections;
- exact target-sample matching (rule="target_match"): draw from the target at
  each node and descend while the draw is a child's token.

Pinned against hand-derived closed forms, against the pinned single-residual
walk (chains) and greedy walk (one-hot targets), and against the
distribution-preservation property each rule has: with the children's tokens
drawn i.i.d. from q the iterated rule emits p-distributed tokens, and the
matching rule does so for any tree.  The single-residual rule, a plausible
mistake for the iterated one, fails the same frequency test."""
import numpy as np
import pytest

import oracle


def _tree(tok, parent, rank):
    tok = np.array(tok, np.int32)
    parent = np.array(parent, np.int32)
    depth = np.zeros(len(tok), np.int32)
    for i in range(1, len(tok)):
        depth[i] = depth[parent[i]] + 1
    return oracle.Tree(tok, parent, depth, np.array(rank, np.int32), np.zeros(len(tok), np.float32), len(tok))


def _star(tokens):
    """Root with one leaf child per token, tested in the given order."""
    k = len(tokens)
    return _tree([-1] + list(tokens), [-1] + [0] * k, [-1] + list(range(k)))


def _chain(tokens):
    n = len(tokens) + 1
    return _tree([-1] + list(tokens), list(range(-1, n - 1)), [-1] + [0] * (n - 1))


def _log32(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _walk(rule, t, p_rows, q_rows, u, L, Mmax):
    """p_rows: [Mmax, V] target log-probabilities (normaliser 0); q_rows: [L, V] drafter log-probabilities."""
    return oracle.verify_t1(t, p_rows, q_rows, np.zeros(L, np.float32), u, L, Mmax,
                            lse_in=np.zeros(Mmax, np.float32), rule=rule)


# ---------------------------------------------------------------------------
# iterated residual: hand-derived closed forms
# ---------------------------------------------------------------------------
def test_iter_residual_fractional_second_acceptance():
    # p = (.4, .3, .2, .1), q = (.1, .35, .15, .4); children D then C.
    # D is accepted with p(D)/q(D) = 1/4.  After rejecting D:
    #   [p - q]_+ = (.3, 0, .05, 0), sum .35  ->  r_1 = (6/7, 0, 1/7, 0)
    # so C is accepted with r_1(C)/q(C) = (1/7)/.15 = 20/21, and after rejecting
    # C too, r_2 = [r_1 - q]_+ normalised = (1, 0, 0, 0): the draw is A.
    p, q = [0.4, 0.3, 0.2, 0.1], [0.1, 0.35, 0.15, 0.4]
    t = _star([3, 2])
    rows = np.stack([_log32(p)] * 3)
    qr = _log32(q)[None, :]
    grid = (np.arange(21000) + 0.5) / 21000
    acc_c = 0
    for uc in grid:
        u = np.array([[0.0, 0.9999, uc], [0.5, 0.5, 0.5]], np.float32)  # D always rejected (u >= 1/4)
        acc, alen, nxt, _ = _walk("iter_residual", t, rows, qr, u, 1, 3)
        if alen == 1:
            assert acc[1] == 2
            acc_c += 1
        else:
            assert nxt == 0
    assert abs(acc_c - 20000) <= 2, acc_c
    # the single-residual rule tests C against p instead: ratio .2/.15 >= 1, always accepted
    u = np.array([[0.0, 0.9999, 0.99], [0.5, 0.5, 0.5]], np.float32)
    assert _walk("ratio", t, rows, qr, u, 1, 3)[1] == 1
    assert _walk("iter_residual", t, rows, qr, u, 1, 3)[1] == 0


def test_iter_residual_replacement_after_two_rejections():
    # p = (.4, .3, .2, .1), q = (.1, .2, .3, .4); children D then C.
    # r_1 = [p - q]_+ / .4 = (.75, .25, 0, 0); C has r_1(C) = 0: always rejected;
    # r_2 = [r_1 - q]_+ / .7 = (.65, .05, 0, 0) / .7 = (13/14, 1/14, 0, 0).
    # (The single-residual rule would draw from r_1: A with 3/4.)
    p, q = [0.4, 0.3, 0.2, 0.1], [0.1, 0.2, 0.3, 0.4]
    t = _star([3, 2])
    rows = np.stack([_log32(p)] * 3)
    qr = _log32(q)[None, :]
    got = {"iter_residual": [], "ratio": []}
    for ur in (np.arange(14000) + 0.5) / 14000:
        for rule in got:
            u = np.array([[0.0, 0.9999, 0.9], [ur, 0.5, 0.5]], np.float32)
            acc, alen, nxt, _ = _walk(rule, t, rows, qr, u, 1, 3)
            assert alen == 0
            got[rule].append(nxt)
    it = np.bincount(got["iter_residual"], minlength=4)
    assert abs(it[0] - 13000) <= 2 and abs(it[1] - 1000) <= 2 and it[2] == 0 and it[3] == 0, it
    one = np.bincount(got["ratio"], minlength=4)
    assert abs(one[0] - 10500) <= 2 and abs(one[1] - 3500) <= 2, one


def test_iter_residual_equals_single_residual_on_chains():
    # one child per node: the rules coincide bit for bit
    rng = np.random.default_rng(5)
    V, L = 40, 5
    for trial in range(40):
        toks = rng.integers(0, V, L).tolist()
        t = _chain(toks)
        tgt = (rng.standard_normal((L + 1, V)) * 2).astype(np.float32)
        x = (rng.standard_normal((L, V)) * 2).astype(np.float32)
        if trial % 2:
            for d in range(L):  # make acceptance likely
                tgt[d, toks[d]] += 4.0
                x[d, toks[d]] += 4.0
        dl = np.array([np.logaddexp.reduce(r.astype(np.float64)) for r in x], np.float32)
        u = rng.random((2, L + 1)).astype(np.float32)
        a = oracle.verify_t1(t, tgt, x, dl, u, L, L + 1, rule="ratio")
        b = oracle.verify_t1(t, tgt, x, dl, u, L, L + 1, rule="iter_residual")
        assert a[0].tolist() == b[0].tolist() and a[1:3] == b[1:3], trial


@pytest.mark.parametrize("rule,lossless", [("iter_residual", True), ("ratio", False)])
def test_iter_residual_preserves_p_for_iid_candidates(rule, lossless):
    # Candidates c_1..c_3 drawn i.i.d. from q (repeats allowed): the iterated
    # rule emits tokens distributed exactly as p; testing every child against
    # p alone does not.
    p = np.array([0.1, 0.2, 0.3, 0.4])
    q = np.array([0.4, 0.3, 0.2, 0.1])
    rows = np.stack([_log32(p)] * 4)
    qr = _log32(q)[None, :]
    rng = np.random.default_rng(99)
    n = 40_000
    cq = np.cumsum(q)
    counts = np.zeros(4, np.int64)
    for _ in range(n):
        toks = np.searchsorted(cq, rng.random(3), side="right").clip(0, 3).tolist()
        u = np.zeros((2, 4), np.float32)
        u[0, 1:] = rng.random(3)
        u[1, 0] = rng.random()
        acc, alen, nxt, _ = _walk(rule, _star(toks), rows, qr, u, 1, 4)
        counts[toks[acc[1] - 1] if alen == 1 else nxt] += 1
    freq = counts / n
    sigma = np.sqrt(p * (1 - p) / n)
    dev = np.abs(freq - p) / sigma
    if lossless:
        assert np.all(dev <= 3.5), (freq, p)
    else:
        assert np.max(dev) > 10, (freq, p)


# ---------------------------------------------------------------------------
# exact target-sample matching
# ---------------------------------------------------------------------------
def test_target_match_draws_by_inverse_cdf_and_descends_on_match():
    # root with children B, D (tokens 1, 3); p_root = (.4, .3, .2, .1):
    # a draw of B or D descends, A or C is emitted.
    p = [0.4, 0.3, 0.2, 0.1]
    t = _tree([-1, 1, 3], [-1, 0, 0], [-1, 0, 1])
    rows = np.stack([_log32(p), _log32([0, 0, 1.0, 0]), _log32([0, 0, 0, 1.0])])
    first = []
    for u1 in (np.arange(10000) + 0.5) / 10000:
        u = np.array([[0.0, 0.0, 0.0], [u1, 0.5, 0.5]], np.float32)
        acc, alen, nxt, _ = oracle.verify_target_match(t, rows, u, 1, 3, lse_in=np.zeros(3, np.float32))
        if alen == 1:
            assert acc[1] in (1, 2) and nxt == (2 if acc[1] == 1 else 3)  # bonus from the one-hot child row
            first.append(int(t.tok[acc[1]]))
        else:
            first.append(nxt)
    c = np.bincount(first, minlength=4)
    assert all(abs(int(c[i]) - int(p[i] * 10000)) <= 2 for i in range(4)), c


def test_target_match_equals_greedy_walk_for_one_hot_targets():
    rng = np.random.default_rng(8)
    V, L = 13, 5
    for trial in range(20):
        x = (rng.standard_normal((L, V)) * 1.5).astype(np.float32)
        _, _, ids, lps = oracle.candidates(x, 3)
        t = oracle.ddtree(lps, ids, 25).trimmed()
        tgt = np.full((t.n, V), -1e4, np.float32)
        for n in range(t.n):
            kids = [int(t.tok[c]) for c in range(1, t.n) if t.parent[c] == n]
            # follow a child most of the time, else a token outside the tree
            choice = kids[rng.integers(len(kids))] if kids and rng.random() < 0.8 else int(rng.integers(V))
            tgt[n, choice] = 0.0
        u = rng.random((2, t.n)).astype(np.float32)
        a = oracle.verify_target_match(t, tgt, u, L, t.n)
        g = oracle.verify_greedy(t, tgt, L)
        assert a[0].tolist() == g[0].tolist() and a[1] == g[1] and a[2] == g[2], trial


def test_target_match_emits_target_samples_along_the_path():
    # first token ~ p_root and, given that it matched child c, the second ~ p_c
    V = 5
    rng = np.random.default_rng(31)
    t = _tree([-1, 0, 2, 4], [-1, 0, 0, 1], [-1, 0, 1, 0])
    P = rng.dirichlet(np.ones(V) * 2, size=4)
    rows = np.stack([_log32(r) for r in P])
    n = 30_000
    first = np.zeros(V, np.int64)
    second = np.zeros(V, np.int64)
    n_first0 = 0
    for _ in range(n):
        u = np.zeros((2, 4), np.float32)
        u[1] = rng.random(4)
        acc, alen, nxt, _ = oracle.verify_target_match(t, rows, u, 2, 4, lse_in=np.zeros(4, np.float32))
        f = int(t.tok[acc[1]]) if alen >= 1 else nxt
        first[f] += 1
        if alen >= 1 and acc[1] == 1:  # matched token 0: the next token comes from row 1
            n_first0 += 1
            second[int(t.tok[acc[2]]) if alen == 2 else nxt] += 1
    for cnt, tot, pr in ((first, n, P[0]), (second, n_first0, P[1])):
        freq = cnt / tot
        sigma = np.sqrt(pr * (1 - pr) / tot)
        assert np.all(np.abs(freq - pr) <= 3.5 * sigma), (freq, pr)


# ---------------------------------------------------------------------------
# T=1 against the normalised DARTree proposal q~(. | parent token)
# ---------------------------------------------------------------------------
def test_markov_walk_without_term_is_the_plain_walk():
    rng = np.random.default_rng(21)
    V, L, K = 30, 4, 3
    for trial in range(25):
        x = (rng.standard_normal((L, V)) * 1.5).astype(np.float32)
        l32, _, ids, lps = oracle.candidates(x, K)
        t = oracle.ddtree(lps, ids, 12).trimmed()
        tgt = (rng.standard_normal((t.n, V)) * 1.5).astype(np.float32)
        u = rng.random((2, t.n)).astype(np.float32)
        zero_U = np.zeros((V, 2), np.float32)
        a = oracle.verify_t1(t, tgt, x, l32, u, L, t.n)
        b = oracle.verify_t1_markov(t, tgt, x, l32, zero_U, zero_U, 5, np.zeros((L, K), np.float32), u, L, t.n)
        assert a[0].tolist() == b[0].tolist() and a[1:3] == b[1:3], trial


def _qtilde(x_row, U, Vt, u, z):
    lp = x_row.astype(np.float64) - np.logaddexp.reduce(x_row.astype(np.float64))
    return np.exp(lp + Vt.astype(np.float64) @ U[u].astype(np.float64) - z)


@pytest.mark.parametrize("proposal,lossless", [("markov", True), ("plain", False)])
def test_markov_walk_preserves_p_when_the_child_is_drawn_from_q_tilde(proposal, lossless):
    # one child under the root, its token drawn from q~(. | root token); the
    # walk with the corrected proposal emits p; the plain marginal does not
    V, R, root = 6, 2, 4
    rng = np.random.default_rng(5)
    x = np.array([[1.0, 0.5, 0.0, -0.5, 0.2, 0.8]], np.float32)
    U = (rng.standard_normal((V, R)) * 1.5).astype(np.float32)
    Vt = (rng.standard_normal((V, R)) * 1.5).astype(np.float32)
    ids = np.arange(V, dtype=np.int32)[None, :1]
    z = oracle.markov_norm(x, ids, U, Vt, root)
    qt = _qtilde(x[0], U, Vt, root, float(z[0, 0]))
    assert abs(qt.sum() - 1) < 1e-5  # the exact normaliser makes q~ a probability
    p = np.array([0.05, 0.3, 0.1, 0.25, 0.2, 0.1])
    rows = np.stack([np.log(p).astype(np.float32)] * 2)
    l32 = np.array([np.logaddexp.reduce(x[0].astype(np.float64))], np.float32)
    n = 30_000
    counts = np.zeros(V, np.int64)
    cq = np.cumsum(qt)
    Uw = U if proposal == "markov" else np.zeros_like(U)
    zw = z if proposal == "markov" else np.zeros_like(z)
    for _ in range(n):
        tok = int(min(np.searchsorted(cq, rng.random(), side="right"), V - 1))
        t = oracle.Tree(np.array([-1, tok], np.int32), np.array([-1, 0], np.int32), np.array([0, 1], np.int32),
                        np.array([-1, 0], np.int32), np.zeros(2, np.float32), 2)
        u = rng.random((2, 2)).astype(np.float32)
        acc, alen, nxt = oracle.verify_t1_markov(t, rows, x, l32, Uw, Vt, root, zw, u, 1, 2,
                                                 lse_in=np.zeros(2, np.float32))
        counts[tok if alen == 1 else nxt] += 1
    dev = np.abs(counts / n - p) / np.sqrt(p * (1 - p) / n)
    if lossless:
        assert np.all(dev <= 3.5), (counts / n, p)
    else:
        assert np.max(dev) > 10, (counts / n, p)


def test_markov_walk_uses_the_parents_own_normaliser():
    # The proposal below a node u is q~(. | tok(u)) normalised by u's own row of
    # the normalisers (its position, its candidate rank).  Root -> u (token 1, the
    # rank-1 candidate of position 1, accepted with certainty) -> one child drawn
    # from q~(. | 1): the token at position 2 must follow p.  The rank-0
    # candidate (token 3) has another normaliser, which would bias it.
    V, R, L, root = 6, 2, 2, 4
    rng = np.random.default_rng(9)
    x = np.array([[0.3, 0.9, -0.2, 1.1, 0.0, -0.4],
                  [1.0, 0.5, 0.0, -0.5, 0.2, 0.8]], np.float32)
    U = (rng.standard_normal((V, R)) * 1.5).astype(np.float32)
    Vt = (rng.standard_normal((V, R)) * 1.5).astype(np.float32)
    ids = np.array([[3, 1], [0, 1]], np.int32)
    z = oracle.markov_norm(x, ids, U, Vt, root)
    assert abs(float(z[1, 0]) - float(z[1, 1])) > 0.2  # the two parents' normalisers differ
    qt = _qtilde(x[1], U, Vt, 1, float(z[1, 1]))
    assert abs(qt.sum() - 1) < 1e-5
    p = np.array([0.05, 0.3, 0.1, 0.25, 0.2, 0.1])
    sure = np.full(V, -30.0, np.float32)
    sure[1] = 0.0  # the root's target takes token 1: u is always accepted
    rows = np.stack([sure, np.log(p).astype(np.float32), np.log(np.full(V, 1 / V)).astype(np.float32)])
    l32 = np.array([np.logaddexp.reduce(r.astype(np.float64)) for r in x], np.float32)
    n = 30_000
    counts = np.zeros(V, np.int64)
    cq = np.cumsum(qt)
    for _ in range(n):
        tok = int(min(np.searchsorted(cq, rng.random(), side="right"), V - 1))
        t = _tree([-1, 1, tok], [-1, 0, 1], [-1, 1, 0])
        u = rng.random((2, 3)).astype(np.float32)
        acc, alen, nxt = oracle.verify_t1_markov(t, rows, x, l32, U, Vt, root, z, u, L, 3,
                                                 lse_in=np.zeros(3, np.float32))
        assert alen >= 1
        counts[tok if alen == 2 else nxt] += 1
    dev = np.abs(counts / n - p) / np.sqrt(p * (1 - p) / n)
    assert np.all(dev <= 3.5), (counts / n, p)
