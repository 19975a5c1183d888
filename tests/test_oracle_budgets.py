"""Pins of the oracle's budget policies (CPU only).

- DARTree (fixed): the budget spread uniformly over the depths ([DARTree]
  experimental setup: 4 nodes per layer for B = 64 over 16 depths), feeding
  per-depth widths to the DARTree supertree;
- SABA ([GRAFT] "State-aware budget allocation"): B_t = argmax a*sqrt(B) /
  (B*c_verify + c_fixed), which is c_fixed / c_verify whatever the state, and
  the state features conf, degen, hist, a by hand."""
import itertools

import numpy as np
import pytest

import oracle


def test_uniform_widths_page_figure_and_spread():
    assert oracle.uniform_widths(64, 16).tolist() == [4] * 16
    for B, L in itertools.product(range(1, 200, 7), range(1, 33)):
        if B < L:
            continue
        w = oracle.uniform_widths(B, L)
        assert w.sum() == B and w.max() - w.min() <= 1
        assert np.all(np.diff(w) <= 0)  # the extra nodes go to the shallowest depths


def _layers(t):
    out = {}
    for v in range(1, t.n):
        out.setdefault(int(t.depth[v]), []).append(v)
    return out


@pytest.mark.parametrize("B,L,K", [(64, 16, 8), (22, 5, 6), (9, 3, 4)])
def test_dartree_fixed_keeps_the_best_w_d_children_per_depth(B, L, K):
    rng = np.random.default_rng(B + L)
    x = (rng.standard_normal((L, 60)) * 2).astype(np.float32)
    _, _, ids, lps = oracle.candidates(x, K)
    U = (rng.standard_normal((60, 4)) * 0.3).astype(np.float32)
    Vt = (rng.standard_normal((60, 4)) * 0.3).astype(np.float32)
    w = oracle.uniform_widths(B, L)
    Wmax = int(w.max())
    t, info, _ = oracle.dartree(lps, ids, U, Vt, 3, Wmax, 0.0, B, Mmax=B + 1, widths=w)
    # the whole supertree is kept (its size is at most B)
    assert t.n - 1 == info["supertree_size"] <= B
    lay = _layers(t)
    prev = [0]
    for d in range(1, L + 1):
        # every child of the kept parents, scored as the supertree does
        E = oracle.markov_table(ids, U, Vt, 3)
        kids = []
        for p in prev:
            pr = 0 if p == 0 else int(t.rank[p])
            for j in range(K):
                tj = np.float32(lps[d - 1, j]) + np.float32(E[d - 1, pr, j])
                kids.append(float(np.float32(np.float32(t.score[p]) + np.float32(tj))))
        kids.sort(reverse=True)
        got = sorted((float(t.score[v]) for v in lay.get(d, [])), reverse=True)
        assert len(got) == min(int(w[d - 1]), len(kids)), d
        assert got == kids[:len(got)], d
        prev = lay.get(d, [])
    # equal widths: the same as DARTree with W = B / L
    if B % L == 0:
        t2, _, _ = oracle.dartree(lps, ids, U, Vt, 3, B // L, 0.0, B, Mmax=B + 1)
        assert t2.n == t.n and np.array_equal(t2.tok[:t.n], t.tok[:t.n]) and np.array_equal(t2.parent[:t.n],
                                                                                             t.parent[:t.n])


@pytest.mark.parametrize("cv,cf,want", [(0.5, 40.0, 80), (0.25, 16.0, 64), (2.0, 300.0, 150), (1.0, 7.0, 7)])
def test_saba_budget_is_c_fixed_over_c_verify(cv, cf, want):
    # d/dB [a sqrt(B) / (B cv + cf)] = 0  <=>  B cv + cf = 2 B cv  <=>  B = cf / cv
    st = oracle.SabaState(8)
    b, _ = oracle.saba(np.zeros(4, np.float32), None, st, -1, cv, cf, 1, 1024)
    assert b == want
    # the state cannot move it: a cancels
    for prev in (0, 3, 15, 1, 9):
        b2, s = oracle.saba(np.full(4, -2.0, np.float32), None, st, prev, cv, cf, 1, 1024)
        assert b2 == want and s[3] >= 1.0


def test_saba_budget_clamps_to_the_range():
    st = oracle.SabaState(4)
    assert oracle.saba(np.zeros(2, np.float32), None, st, -1, 0.01, 5000.0, 16, 256)[0] == 256
    assert oracle.saba(np.zeros(2, np.float32), None, st, -1, 10.0, 1.0, 16, 256)[0] == 16


def test_saba_takes_the_smallest_budget_on_ties():
    # The reading: the smallest B among equal scores.  With c_fixed = 0 the
    # objective a sqrt(B) / (B c_verify) falls with B, so the range's first
    # budget is the maximum; evaluated in fp32, budgets past 2^24 share float
    # values (2^25, 2^25 + 1 and 2^25 + 2 all become 2^25) and tie with it.
    st = oracle.SabaState(2)
    lo = 1 << 25
    assert oracle.saba(np.zeros(2, np.float32), None, st, -1, 1.0, 0.0, lo, lo + 3)[0] == lo
    # c_fixed / c_verify = 1000.5 puts the optimum between 1000 and 1001, whose
    # fp32 scores are equal (checked here with numpy's float32 arithmetic)
    f = np.float32
    u = [f(f(1.0) * np.sqrt(f(b))) / f(f(b) * f(1.0) + f(1000.5)) for b in (1000, 1001)]
    assert u[0] == u[1]
    assert oracle.saba(np.zeros(2, np.float32), None, st, -1, 1.0, 1000.5, 1, 1024)[0] == 1000


def test_saba_state_by_hand():
    # conf: top probabilities 0.5 and 0.25 -> 0.375
    # degen: h = (1,0), (1,0), (0,1): r = (1, 0), mean 0.5, growth 0 - 1 -> -0.5
    # history w = 2: lengths 3, 5, 7 pushed -> window (5, 7): hist 6, a = mean(l + 1) = 7
    st = oracle.SabaState(2)
    hid = np.array([[1, 0], [1, 0], [0, 1]], np.float32)
    top = np.log(np.array([0.5, 0.25, 0.375])).astype(np.float32)
    _, s0 = oracle.saba(top, hid, st, -1, 1.0, 10.0, 1, 64)
    assert s0[2] == 0.0 and s0[3] == 1.0  # no history yet
    for prev in (3, 5, 7):
        _, s = oracle.saba(top, hid, st, prev, 1.0, 10.0, 1, 64)
        if prev == 3:  # one round recorded, fewer than w: hist 3, a = 3 + 1
            assert s[2] == 3.0 and s[3] == 4.0
    assert abs(s[0] - (0.5 + 0.25 + 0.375) / 3) < 1e-6
    assert abs(s[1] - (-0.5)) < 1e-6
    assert s[2] == 6.0 and s[3] == 7.0
    assert st.count[0] == 3 and sorted(st.ring.tolist()) == [5, 7]
