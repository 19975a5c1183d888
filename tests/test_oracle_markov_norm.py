"""Pins of the oracle's full-vocabulary normalised DARTree correction.

[DARTree] "Causal correction": the corrected drafter distribution q~ is a
probability over the vocabulary, so its log-normaliser for a parent token u at
position d is log Z_d(u) = log sum_v exp(lp_d(v) + <U[u], Vt[v]>).  These tests
pin oracle.markov_norm and the normalised selection to facts that do not come
from retyping that formula: a hand-worked V = 3 case, special cases, an
invariance, bounds, and Lemma 1's hypothesis becoming true."""
import math

import numpy as np
import pytest

import oracle



def _golden_case():
    # V = 3 tokens, R = 2, L = 2 positions, K = 2 candidates per position
    x = np.array([[0.0, 0.0, 0.0], [1.0, 0.0, 0.0]], np.float32)
    U = np.array([[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]], np.float32)
    Vt = np.array([[0.5, 0.0], [0.0, 0.25], [0.0, 0.0]], np.float32)
    ids = np.array([[0, 1], [0, 2]], np.int32)
    return x, U, Vt, ids


def test_hand_worked_three_token_case():
    x, U, Vt, ids = _golden_case()
    z = oracle.markov_norm(x, ids, U, Vt, root_tok=1)
    e = math.e
    # position 0, parent = root token 1: terms m(1, .) = (0, 0.25, 0) on x = 0
    assert z[0, 0] == pytest.approx(math.log((2 + math.exp(0.25)) / 3), abs=1e-7)
    assert z[0, 1] == 0.0  # only the root row has a term at position 0
    # position 1, parents = candidates of position 0 (tokens 0 and 1), x = (1, 0, 0)
    assert z[1, 0] == pytest.approx(math.log(math.exp(1.5) + 2) - math.log(e + 2), abs=1e-7)
    assert z[1, 1] == pytest.approx(math.log(e + math.exp(0.25) + 1) - math.log(e + 2), abs=1e-7)
    # no root token: position 0 has no term at all
    z2 = oracle.markov_norm(x, ids, U, Vt, root_tok=-1)
    assert np.all(z2[0] == 0.0) and np.array_equal(z2[1], z[1])
    # one row at a time gives the same values
    for r in range(4):
        zr = oracle.markov_norm(x, ids, U, Vt, root_tok=1, only_row=r)
        assert zr.reshape(-1)[r] == z.reshape(-1)[r]


def _random(seed, L=3, V=50, K=4, R=8, scale=2.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((L, V)) * scale).astype(np.float32)
    U = (rng.standard_normal((V, R)) * 0.3).astype(np.float32)
    Vt = (rng.standard_normal((V, R)) * 0.3).astype(np.float32)
    ids = np.stack([rng.permutation(V)[:K] for _ in range(L)]).astype(np.int32)
    return x, U, Vt, ids


def test_zero_table_gives_zero():
    x, U, Vt, ids = _random(1)
    z = oracle.markov_norm(x, ids, np.zeros_like(U), Vt, root_tok=5)
    assert np.max(np.abs(z)) < 1e-7  # sum of exp(lp) is 1


def test_one_token_vocabulary_gives_its_own_term():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 1)).astype(np.float32)
    U = rng.standard_normal((1, 8)).astype(np.float32)
    Vt = rng.standard_normal((1, 8)).astype(np.float32)
    ids = np.zeros((3, 1), np.int32)
    z = oracle.markov_norm(x, ids, U, Vt, root_tok=0)
    own = float(np.dot(U[0].astype(np.float64), Vt[0].astype(np.float64)))  # lp = 0 for the only token
    assert np.allclose(z, own, atol=1e-6)


def test_constant_shift_of_every_term_shifts_the_normaliser():
    x, U, Vt, ids = _random(3)
    U = U.copy()
    U[:, 0] = 1.0
    z = oracle.markov_norm(x, ids, U, Vt, root_tok=7)
    Vs = Vt.copy()
    Vs[:, 0] += 0.75  # every <U[u], Vt[v]> grows by 0.75
    zs = oracle.markov_norm(x, ids, U, Vs, root_tok=7)
    has = np.ones_like(z, bool)
    has[0, 1:] = False  # rows without a term stay 0
    assert np.allclose(zs[has] - z[has], 0.75, atol=2e-6)
    assert np.all(zs[~has] == 0.0)


def test_bounds_and_normalisation():
    x, U, Vt, ids = _random(4, V=200)
    z = oracle.markov_norm(x, ids, U, Vt, root_tok=11)
    L, V = x.shape
    for d in range(L):
        xd = x[d].astype(np.float64)
        lp = xd - (xd.max() + np.log(np.exp(xd - xd.max()).sum()))
        for i in range(ids.shape[1]):
            u = 11 if d == 0 else ids[d - 1, i]
            if d == 0 and i > 0:
                continue
            a = lp + U[u].astype(np.float64) @ Vt.astype(np.float64).T
            assert a.max() - 1e-6 <= z[d, i] <= a.max() + np.log(V) + 1e-6
            assert abs(np.exp(a - np.float64(z[d, i])).sum() - 1.0) < 1e-6


def test_normalised_selection_reduces_to_plain_for_zero_table():
    x, U, Vt, ids = _random(5, L=4, V=40, K=5)
    lse64, l32, cid, lps = oracle.candidates(x, 5)
    Z0 = np.zeros_like(U)
    z = oracle.markov_norm(x, cid, Z0, Vt, root_tok=3)
    a, _, _ = oracle.dartree(lps, cid, Z0, Vt, 3, W=6, beta=-0.25, B=20)
    b, _, _ = oracle.dartree(lps, cid, Z0, Vt, 3, W=6, beta=-0.25, B=20, znorm=z)
    for f in ("tok", "parent", "depth", "rank", "score"):
        assert np.array_equal(getattr(a, f)[:a.n], getattr(b, f)[:b.n]), f


def test_normalised_correction_satisfies_lemma_one():
    # an unnormalised Markov term can raise a child above its parent (Lemma 1's
    # hypothesis fails); the normalised q~ <= 1 never does, so TopB(S) is the
    # best-first tree with no violating edge
    rng = np.random.default_rng(6)
    L, V, K = 5, 60, 6
    x = (rng.standard_normal((L, V)) * 0.3).astype(np.float32)
    x[:, 0] += 6.0  # a confident token: lp close to 0
    U = (rng.standard_normal((V, 8)) * 0.6).astype(np.float32)
    Vt = (rng.standard_normal((V, 8)) * 0.6).astype(np.float32)
    _, _, cid, lps = oracle.candidates(x, K)
    _, info_raw, _ = oracle.dartree(lps, cid, U, Vt, 0, W=8, beta=0.0, B=30)
    assert info_raw["violations"] > 0
    z = oracle.markov_norm(x, cid, U, Vt, root_tok=0)
    _, info, _ = oracle.dartree(lps, cid, U, Vt, 0, W=8, beta=0.0, B=30, znorm=z)
    assert info["violations"] == 0 and info["topb_equals_bestfirst"]
