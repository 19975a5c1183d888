"""Pins for the end-to-end selection check (oracle.selection_check), on the CPU.

The check claims that a tree selected from a stage-1 table whose log-probs are
within 1e-5 of the oracle's differs from the oracle's tree only by near-ties,
within the tolerance it derives from the path sums.  That claim is tested here
without any GPU: the oracle itself selects from a perturbed table (every
position's log-probs moved by the same amount, below 1e-5, as a different
normaliser would move them), and the check must explain every difference.  A
perturbation far beyond the contract, and a node order broken on purpose, must
be reported.
"""
import numpy as np
import pytest

import oracle

EPS = 1e-5


def _table(rng, L, V, K, scale, dtype=np.float32):
    x = (rng.standard_normal((L, V)) * scale).astype(np.float32)
    if dtype == "bf16":  # round to bf16 (nearest even): many exact ties
        b = x.view(np.uint32).astype(np.uint64)
        b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
        x = b.astype(np.uint32).view(np.float32)
    _, _, ids, lps = oracle.candidates(x, K)
    return x, ids, lps


def _perturb(rng, lps, eps):
    """Every position's log-probs moved by one offset in [-eps, eps] (fp32)."""
    d = rng.uniform(-eps, eps, size=(lps.shape[0], 1)).astype(np.float32)
    out = (lps - d).astype(np.float32)
    assert np.max(np.abs(out.astype(np.float64) - lps)) <= EPS
    return out


def _assert_explained(rep):
    assert rep["mismatches"] == [], rep["mismatches"][:3]
    assert rep["order_mismatches"] == 0
    assert rep["score_err_viol"] == 0


def test_rescoring_reproduces_the_oracle_scores_in_every_mode():
    rng = np.random.default_rng(1)
    x, ids, lps = _table(rng, 6, 400, 8, 2.0)
    U = (rng.standard_normal((400, 8)) * 0.3).astype(np.float32)
    Vt = (rng.standard_normal((400, 8)) * 0.3).astype(np.float32)
    E = oracle.markov_table(ids, U, Vt, 5)
    z = oracle.markov_norm(x, ids, U, Vt, 5)
    cases = [
        ("ddtree", oracle.ddtree(lps, ids, 40), {}),
        ("talon", oracle.talon(lps, ids, 4, float(np.float32(np.log(0.05))), 40), {}),
        ("dartree", oracle.dartree(lps, ids, U, Vt, 5, 6, -0.25, 30)[0], dict(E=E, beta=-0.25, root_term=True)),
        ("dartree", oracle.dartree(lps, ids, U, Vt, 5, 6, 0.0, 30, znorm=z)[0],
         dict(E=E, znorm=z, root_term=True)),
        ("heap", oracle.heap_select(lps, ids, 40, E=E), dict(E=E)),
        ("heap", oracle.heap_select(lps, ids, 40, E=E, znorm=z), dict(E=E, znorm=z)),
    ]
    for mode, t, kw in cases:
        t = t.trimmed()
        s, _, _ = oracle.path_scores(t, lps, mode, **kw)
        assert np.array_equal(s[1:].view(np.uint32), t.score[1:].view(np.uint32)), mode
        rep = oracle.selection_check(t, t, lps, mode, got_scores=t.score, **kw)
        assert rep["differing"] == 0 and rep["order_swaps"] == 0 and rep["score_err_max"] == 0.0


# scales: spiky, bf16 with exact ties, and nearly flat fp32 rows (path scores
# packed densely enough that a shift below 1e-5 moves selections)
@pytest.mark.parametrize("scale,dtype,B", [(3.0, "f32", 64), (0.3, "bf16", 64), (0.0003, "f32", 120)])
def test_ddtree_perturbed_tables_differ_only_by_near_ties(scale, dtype, B):
    rng = np.random.default_rng(int(scale * 100) + B)
    total = 0
    for trial in range(30):
        _, ids, lps = _table(rng, 8, 600, 16, scale, dtype)
        want = oracle.ddtree(lps, ids, B).trimmed()
        got = oracle.ddtree(_perturb(rng, lps, 9e-6), ids, B).trimmed()
        rep = oracle.selection_check(got, want, lps, "ddtree", got_scores=got.score)
        _assert_explained(rep)
        total += rep["near_ties"] + rep["order_swaps"]
    if scale < 0.001:  # nearly flat rows: the perturbation must actually move selections
        assert total > 0


@pytest.mark.parametrize("scale,dtype", [(0.4, "bf16"), (0.0003, "f32")])
def test_talon_perturbed_tables_differ_only_by_near_ties(scale, dtype):
    rng = np.random.default_rng(5)
    log_mu = float(np.float32(np.log(0.03)))
    total = 0
    for trial in range(30):
        _, ids, lps = _table(rng, 8, 800, 60, scale, dtype)
        want = oracle.talon(lps, ids, 10, log_mu, 60).trimmed()
        got = oracle.talon(_perturb(rng, lps, 9e-6), ids, 10, log_mu, 60).trimmed()
        rep = oracle.selection_check(got, want, lps, "talon", log_mu=log_mu, got_scores=got.score)
        _assert_explained(rep)
        total += rep["near_ties"]
    if scale < 0.001:
        assert total > 0


@pytest.mark.parametrize("B", [25, 400])
def test_dartree_perturbed_tables_differ_only_by_near_ties(B):
    rng = np.random.default_rng(B)
    total = 0
    for trial in range(20):
        _, ids, lps = _table(rng, 6, 500, 6, 0.0003, "f32")  # nearly flat rows, a weak Markov term
        U = (rng.standard_normal((500, 8)) * 0.003).astype(np.float32)
        Vt = (rng.standard_normal((500, 8)) * 0.003).astype(np.float32)
        E = oracle.markov_table(ids, U, Vt, -1)
        want = oracle.dartree(lps, ids, U, Vt, -1, 8, -0.5, B)[0].trimmed()
        got = oracle.dartree(_perturb(rng, lps, 9e-6), ids, U, Vt, -1, 8, -0.5, B)[0].trimmed()
        rep = oracle.selection_check(got, want, lps, "dartree", E=E, beta=-0.5, got_scores=got.score)
        _assert_explained(rep)
        total += rep["near_ties"]
    assert total > 0


def test_heap_perturbed_tables_differ_only_by_near_ties():
    rng = np.random.default_rng(9)
    for trial in range(20):
        _, ids, lps = _table(rng, 6, 500, 8, 0.3, "bf16")
        U = (rng.standard_normal((500, 8)) * 0.1).astype(np.float32)
        Vt = (rng.standard_normal((500, 8)) * 0.1).astype(np.float32)
        E = oracle.markov_table(ids, U, Vt, -1)
        want = oracle.heap_select(lps, ids, 60, E=E).trimmed()
        got = oracle.heap_select(_perturb(rng, lps, 9e-6), ids, 60, E=E).trimmed()
        _assert_explained(oracle.selection_check(got, want, lps, "heap", E=E, got_scores=got.score))


def test_a_wrong_normaliser_is_reported():
    # one position's log-probs off by 0.5 (a normaliser far beyond 1e-5): the
    # selections differ at nodes far from every cut
    rng = np.random.default_rng(3)
    _, ids, lps = _table(rng, 8, 600, 16, 3.0)
    want = oracle.ddtree(lps, ids, 64).trimmed()
    bad = lps.copy()
    bad[2] += np.float32(0.5)
    got = oracle.ddtree(bad, ids, 64).trimmed()
    rep = oracle.selection_check(got, want, lps, "ddtree", got_scores=got.score)
    assert len(rep["mismatches"]) > 0
    assert rep["score_err_viol"] > 0


def test_a_broken_node_order_is_reported():
    rng = np.random.default_rng(4)
    _, ids, lps = _table(rng, 6, 500, 8, 3.0)
    want = oracle.ddtree(lps, ids, 30).trimmed()
    # swap the first and the last depth-1 node in the listing (parents remapped)
    d1 = [i for i in range(1, want.n) if want.depth[i] == 1]
    a, b = d1[0], d1[-1]
    assert want.score[a] - want.score[b] > 1e-3
    perm = np.arange(want.n)
    perm[a], perm[b] = b, a
    inv = np.argsort(perm)
    got = oracle.Tree(want.tok[perm], np.where(want.parent[perm] >= 0, inv[np.maximum(want.parent[perm], 0)], -1)
                      .astype(np.int32), want.depth[perm], want.rank[perm], want.score[perm], want.n)
    rep = oracle.selection_check(got, want, lps, "ddtree", got_scores=got.score)
    assert rep["differing"] == 0
    assert rep["order_mismatches"] > 0
