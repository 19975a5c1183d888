"""Pins for the CPU oracle, on the CPU: each check ties the oracle to something
other than itself -- values the pages print, closed forms, invariants,
brute-force enumeration written here independently, library routines from
another library.  A planted mistake in the oracle (the printed DDTree
successor condition) must fail one of them."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from speculative_decoding_draft_bf16_gb300 import workloads as wk


# --------------------------------------------------------------------------
# exp_canon: Cody-Waite reduction + degree-7 Taylor/Horner, checked against
# double-precision exp (a different implementation) and for monotonicity.
# --------------------------------------------------------------------------
def _ulp32(x):
    x = np.abs(np.float32(x))
    return float(np.spacing(x))


def test_exp_canon_ulp_error_and_monotone():
    xs = np.concatenate([np.linspace(-86.0, 88.0, 400001, dtype=np.float64),
                         np.linspace(-1.0, 1.0, 100001, dtype=np.float64)]).astype(np.float32)
    xs = np.unique(xs)
    y = oracle.exp_canon(xs)
    ref = np.exp(xs.astype(np.float64))
    ulps = np.abs(y.astype(np.float64) - ref) / np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert ulps.max() <= 2.0, ulps.max()
    assert np.all(np.diff(y) >= 0), "exp_canon must be monotone"
    assert oracle.exp_canon(np.zeros(1))[0] == 1.0
    assert np.all(oracle.exp_canon(-np.abs(xs)) <= 1.0)
    assert oracle.exp_canon(np.array([-87.0]))[0] == 0.0
    assert np.isinf(oracle.exp_canon(np.array([89.0]))[0])


def test_exp_canon_top_of_range_is_finite():
    # e^x stays below FLT_MAX up to ln(FLT_MAX) = 88.72; the range the function
    # states ends at 88.5.  Above 127.5 ln 2 = 88.376 the reduction picks k = 128,
    # whose power of two is not a float, and the value must still be finite.
    xs = np.array([88.3, 88.376, 88.38, 88.4, 88.45, 88.5], dtype=np.float32)
    y = oracle.exp_canon(xs)
    assert np.all(np.isfinite(y)), y
    ref = np.exp(xs.astype(np.float64))
    ulps = np.abs(y.astype(np.float64) - ref) / np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert ulps.max() <= 2.0, ulps
    assert np.all(np.diff(y) > 0)


# --------------------------------------------------------------------------
# Stage 1: log-normaliser and Top-Kc list.
# --------------------------------------------------------------------------
def test_lse_uniform_row_closed_form():
    V = 151936
    for c in (0.0, 3.25, -7.5):
        x = np.full((1, V), c, np.float32)
        lse64, lse32, ids, lps = oracle.candidates(x, 8)
        assert abs(lse64[0] - (c + math.log(V))) < 1e-9
        assert np.all(ids[0] == np.arange(8))  # all equal: smallest ids first
        assert np.all(np.abs(lps[0] + math.log(V)) <= 2 * _ulp32(c + math.log(V)))


def test_lse_shift_invariance_and_normalisation():
    rng = np.random.default_rng(1)
    # multiples of 1/256 below 16 in magnitude: adding 64 is exact in fp32
    x = (np.round(np.clip(rng.standard_normal((3, 5000)) * 3, -15, 15) * 256) / 256).astype(np.float32)
    a64, _, _, _ = oracle.candidates(x, 4)
    b64, _, _, _ = oracle.candidates(x + np.float32(64.0), 4)
    assert np.allclose(b64 - a64, 64.0, atol=1e-9, rtol=0)
    # all of V as the list: the probabilities sum to one
    _, l32, ids, lps = oracle.candidates(x, 5000)
    assert np.allclose(np.exp(lps.astype(np.float64)).sum(1), 1.0, atol=2e-5)
    # lp of each listed token is its logit minus the normaliser
    assert np.allclose(lps, np.take_along_axis(x, ids, 1) - l32[:, None], atol=0, rtol=0)


def test_topk_rank_order_matches_independent_sort():
    # bf16-rounded values tie a lot; the order is logit desc, then id asc
    rng = np.random.default_rng(2)
    x = torch.tensor(rng.standard_normal((4, 3001)) * 3, dtype=torch.float32)
    x = x.to(torch.bfloat16).float().numpy()
    K = 700
    _, _, ids, _ = oracle.candidates(x, K)
    for r in range(x.shape[0]):
        order = np.lexsort((np.arange(x.shape[1]), -x[r]))[:K]
        assert np.array_equal(ids[r], order)


def test_topk_hand_case_ties_by_id():
    x = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, -1.0]], np.float32)
    _, _, ids, _ = oracle.candidates(x, 4)
    assert ids[0].tolist() == [1, 2, 4, 3]


# --------------------------------------------------------------------------
# DDTree: the heap against brute-force enumeration of S_K written here.
# --------------------------------------------------------------------------
def _f32sum(vals):
    s = np.float32(0.0)
    for v in vals:
        s = np.float32(s + np.float32(v))
    return s


def brute_topb(lp, B):
    """All prefixes of S_K, scored left to right in fp32, sorted by
    (score desc, rank tuple asc with prefix first); first B."""
    L, K = lp.shape
    nodes = []
    for d in range(1, L + 1):
        for rho in itertools.product(range(K), repeat=d):
            nodes.append((-float(_f32sum(lp[i, rho[i]] for i in range(d))), rho))
    nodes.sort()
    return [(rho, -s) for s, rho in nodes[:B]]


def tree_descriptors(t):
    """Rank descriptor of every non-root node by walking parents."""
    out = []
    for n in range(1, t.n):
        rho = []
        a = n
        while a != 0:
            rho.append(int(t.rank[a]))
            a = int(t.parent[a])
        out.append(tuple(reversed(rho)))
    return out


def _check_ddtree_vs_brute(lp, ids, B, rule=0):
    t = oracle.ddtree(lp, ids, B, rule=rule)
    want = brute_topb(lp, B)
    got = list(zip(tree_descriptors(t), t.score[1:t.n].tolist()))
    return [(r, float(s)) for r, s in got] == [(r, float(s)) for r, s in want], t


def _tiny_lists(rng, L, K, V, ties):
    x = rng.standard_normal((L, V)) * 2
    if ties:
        x = np.round(x * 2) / 2  # many exact ties
    x = x.astype(np.float32)
    _, _, ids, lps = oracle.candidates(x, K)
    return lps, ids


def test_ddtree_heap_equals_bruteforce_tiny_config():
    # the tiny greedy workload: L=4, V=32, K=4, B=8, fp32 2*N(0,1), seed 0
    wl = wk.tiny_greedy()
    x, _ = wk.draft_logits(wl)
    _, _, ids, lps = oracle.candidates(x[0].numpy(), wl.K)
    ok, t = _check_ddtree_vs_brute(lps, ids, wl.B)
    assert ok
    assert t.n == wl.B + 1


@pytest.mark.parametrize("seed", range(12))
def test_ddtree_heap_equals_bruteforce_random(seed):
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(1, 5))
    K = int(rng.integers(1, 5))
    lps, ids = _tiny_lists(rng, L, K, 7, ties=bool(seed % 2))
    total = sum(K ** d for d in range(1, L + 1))
    for B in (1, 3, 8, total, total + 5):
        ok, t = _check_ddtree_vs_brute(lps, ids, B)
        assert ok, (seed, B)
        assert t.n == min(B, total) + 1


def test_ddtree_two_token_vocab_depth3():
    # the explainer's closing advice: a 2-token vocabulary, depth 3, checked by enumeration
    lp = np.log(np.array([[0.7, 0.3], [0.6, 0.4], [0.9, 0.1]])).astype(np.float32)
    ids = np.array([[0, 1]] * 3, np.int32)
    for B in range(1, 15):
        ok, _ = _check_ddtree_vs_brute(lp, ids, B)
        assert ok, B


def test_ddtree_printed_successor_rule_fails_bruteforce():
    # Planted mistake: the successor condition as printed (first child only when
    # the last rank is the top one) misses prefixes like (2,1); brute force
    # must catch it on a case where such a prefix belongs to the Top-B.
    lp = np.log(np.array([[0.5, 0.49, 0.01], [0.9, 0.05, 0.05]])).astype(np.float32)
    ids = np.array([[0, 1, 2]] * 2, np.int32)
    ok_good, _ = _check_ddtree_vs_brute(lp, ids, 4, rule=0)
    ok_bad, _ = _check_ddtree_vs_brute(lp, ids, 4, rule=1)
    assert ok_good and not ok_bad


def test_ddtree_lemma_sk_full_vocab_enumeration():
    # Lemma (S_K): with K = min(B, V) the tree equals the Top-B over ALL V^d
    # prefixes (K = V = 32, L = 4: 1,082,400 prefixes enumerated with numpy).
    wl = wk.tiny_greedy()
    x, _ = wk.draft_logits(wl)
    x = x[0].numpy()
    B = wl.B
    _, l32, _, _ = oracle.candidates(x, 1)
    lpfull = (x - l32[:, None]).astype(np.float32)  # [L, V] by token id
    L, V = lpfull.shape
    best = []
    for d in range(1, L + 1):
        grids = np.meshgrid(*[np.arange(V)] * d, indexing="ij")
        toks = np.stack([g.reshape(-1) for g in grids], 1)  # lexicographic in token ids
        s = np.zeros(toks.shape[0], np.float32)
        for i in range(d):
            s = (s + lpfull[i, toks[:, i]]).astype(np.float32)
        keep = np.argsort(-s, kind="stable")[:B]
        best += [(-float(s[j]), tuple(toks[j])) for j in keep]
    best.sort()
    want_paths = [p for _, p in best[:B]]
    _, _, ids, lps = oracle.candidates(x, min(B, V))
    t = oracle.ddtree(lps, ids, B)
    got_paths = []
    for n in range(1, t.n):
        path, a = [], n
        while a != 0:
            path.append(int(t.tok[a]))
            a = int(t.parent[a])
        got_paths.append(tuple(reversed(path)))
    # scores are distinct here, so token ids vs ranks cannot reorder ties
    assert sorted(got_paths) == sorted(want_paths)


def _prefix_closed_subsets(nodes, size):
    """All prefix-closed subsets (trees hanging off the root) of a given size."""
    nodes = sorted(nodes, key=lambda r: (len(r), r))
    out = []

    def rec(chosen, frontier):
        if len(chosen) == size:
            out.append(frozenset(chosen))
            return
        for i, f in enumerate(frontier):
            new_front = frontier[i + 1:] + [c for c in nodes if len(c) == len(f) + 1 and c[:-1] == f]
            rec(chosen + [f], new_front)

    rec([], [r for r in nodes if len(r) == 1])
    return out


def test_ddtree_prop1_objective_optimal_tiny():
    # Prop 1: the Top-B prefix set maximises sum_{u in T} q(u) over all
    # prefix-closed sets of size B (q(u) = product of the positions' probs).
    rng = np.random.default_rng(7)
    V = L = 3
    for trial in range(3):
        pr = rng.dirichlet(np.ones(V), size=L)
        lp = np.log(np.sort(pr, 1)[:, ::-1]).astype(np.float32)
        ids = np.tile(np.arange(V, dtype=np.int32), (L, 1))
        nodes = [r for d in range(1, L + 1) for r in itertools.product(range(V), repeat=d)]

        def q(rho):
            return float(np.prod([np.exp(np.float64(lp[i, rho[i]])) for i in range(len(rho))]))

        for B in range(1, 7):
            t = oracle.ddtree(lp, ids, B)
            ours = sum(q(r) for r in tree_descriptors(t))
            best = max(sum(q(r) for r in s) for s in _prefix_closed_subsets(nodes, B))
            assert ours >= best - 1e-12, (trial, B, ours, best)


def test_ddtree_invariants_qwen_like():
    # prefix closure, parents precede children, scores non-increasing in output order
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((16, 20000)) * 3).astype(np.float32)
    x[np.arange(16), rng.integers(0, 20000, 16)] += 8
    x = torch.tensor(x).to(torch.bfloat16).float().numpy()
    _, _, ids, lps = oracle.candidates(x, 64)
    t = oracle.ddtree(lps, ids, 64)
    assert t.n == 65
    assert np.all(np.diff(t.score[1:t.n]) <= 0)
    for n in range(1, t.n):
        p = t.parent[n]
        assert 0 <= p < n
        assert t.depth[n] == t.depth[p] + 1
        assert t.tok[n] == ids[t.depth[n] - 1, t.rank[n]]


# --------------------------------------------------------------------------
# DARTree
# --------------------------------------------------------------------------
def test_dartree_reduces_to_ddtree_without_correction():
    # U = 0 (no Markov term), beta = 0 and W >= K^(L-1): no per-depth pruning,
    # S = S_K, and TopB(S) is the DDTree Top-B (content and order).
    rng = np.random.default_rng(11)
    for trial in range(6):
        L, K = 3, 3
        lps, ids = _tiny_lists(rng, L, K, 6, ties=bool(trial % 2))
        for B in (1, 4, 9, 39):
            d, info, _ = oracle.dartree(lps, ids, None, None, -1, K ** (L - 1) * K, 0.0, B)
            t = oracle.ddtree(lps, ids, B)
            assert d.n == t.n
            for f in ("tok", "parent", "depth", "rank", "score"):
                assert np.array_equal(getattr(d, f)[:d.n], getattr(t, f)[:t.n]), (trial, B, f)
            assert info["topb_equals_bestfirst"]


def test_dartree_markov_term_and_scores():
    # Each node's score increment equals beta + lp + <U[parent tok], Vt[child tok]>
    # (checked in double against numpy's dot; a transposed or mis-indexed
    # operand would fail this).
    rng = np.random.default_rng(5)
    V, L, K, R, W = 50, 5, 4, 8, 6
    x = (rng.standard_normal((L, V)) * 3).astype(np.float32)
    _, _, ids, lps = oracle.candidates(x, K)
    U = (rng.standard_normal((V, R)) * 0.3).astype(np.float32)
    Vt = (rng.standard_normal((V, R)) * 0.3).astype(np.float32)
    root_tok = 17
    beta = -0.25
    d, info, _ = oracle.dartree(lps, ids, U, Vt, root_tok, W, beta, 200)
    assert info["supertree_size"] == min(W, K) + sum(min(W, W * K) for _ in range(L - 1))
    for n in range(1, d.n):
        p = d.parent[n]
        ptok = root_tok if p == 0 else d.tok[p]
        lp = float(lps[d.depth[n] - 1, d.rank[n]])
        m = float(np.dot(U[ptok].astype(np.float64), Vt[d.tok[n]].astype(np.float64)))
        inc = float(d.score[n]) - float(d.score[p])
        assert abs(inc - (lp + m + beta)) < 1e-4


def test_dartree_lemma1_topb_equals_bestfirst_and_beta_counterexample():
    rng = np.random.default_rng(9)
    V, L, K, R, W = 200, 8, 8, 16, 6
    for beta in (0.0, -0.5):
        for trial in range(5):
            x = (rng.standard_normal((L, V)) * 3).astype(np.float32)
            _, _, ids, lps = oracle.candidates(x, K)
            U = (rng.standard_normal((V, R)) * 0.1).astype(np.float32)
            Vt = (rng.standard_normal((V, R)) * 0.1).astype(np.float32)
            for B in (5, 20, 40):
                d, info, _ = oracle.dartree(lps, ids, U, Vt, -1, W, beta, B)
                if info["violations"] == 0:
                    assert info["topb_equals_bestfirst"], (beta, trial, B)
    # beta > 0 can rank a child above its parent (the pages warn the equality
    # may then fail): a two-token chain where the depth bonus outweighs lp.
    lp = np.log(np.array([[0.6, 0.4], [0.99, 0.01]])).astype(np.float32)
    ids = np.array([[0, 1], [0, 1]], np.int32)
    d, info, topb = oracle.dartree(lp, ids, None, None, -1, 2, 0.5, 1)
    assert info["violations"] > 0
    assert not info["topb_equals_bestfirst"]
    # best-first keeps the tree prefix-closed: its single node is at depth 1
    assert d.n == 2 and d.depth[1] == 1


# --------------------------------------------------------------------------
# TALON
# --------------------------------------------------------------------------
def test_talon_hand_computed_case():
    g = read_golden("talon_v4_l3.txt")
    lp = np.array([[float(v) for v in g["log2probs%d" % i][0]] for i in (1, 2, 3)], np.float32)
    ids = np.array([np.lexsort((np.arange(4), -row)) for row in lp], np.int32)
    lp_sorted = np.take_along_axis(lp, ids, 1)
    t = oracle.talon(lp_sorted, ids, int(g["k"][0][0]), float(g["log2mu"][0][0]), int(g["N"][0][0]))
    want = [[float(v) for v in row] for row in g["node"]]
    assert t.n == len(want) + 1
    for row in want:
        n, tok, par, dep, rnk, sc = int(row[0]), *[int(v) for v in row[1:5]], row[5]
        assert (t.tok[n], t.parent[n], t.depth[n], t.rank[n], float(t.score[n])) == (tok, par, dep, rnk, sc)


def _talon_case(rng, V, L, N, k, mu, flat=False):
    x = rng.standard_normal((L, V)) * (0.01 if flat else 3)
    x = x.astype(np.float32)
    Kc = min(N, V)
    _, _, ids, lps = oracle.candidates(x, V)
    return lps, ids, Kc, np.float32(math.log(mu))


def test_talon_invariants_and_full_list_equivalence():
    rng = np.random.default_rng(21)
    for trial in range(10):
        V, L, N, k, mu = 40, 5, int(rng.integers(3, 30)), int(rng.integers(1, 6)), float(rng.uniform(0.01, 0.5))
        k = min(k, N)
        lps, ids, Kc, log_mu = _talon_case(rng, V, L, N, k, mu)
        t_full = oracle.talon(lps, ids, k, log_mu, N)
        t = oracle.talon(lps[:, :Kc], ids[:, :Kc], k, log_mu, N)
        for f in ("tok", "parent", "depth", "rank", "score"):
            assert np.array_equal(getattr(t, f)[:t.n], getattr(t_full, f)[:t_full.n])
        assert t.n - 1 <= N
        d1 = [n for n in range(1, t.n) if t.depth[n] == 1]
        assert sorted(t.rank[d1].tolist()) == list(range(min(k, N)))
        # every node of depth >= 2 passes its layer's gate: s >= max_pool + log mu
        for d in range(2, L + 1):
            par = [n for n in range(1, t.n) if t.depth[n] == d - 1]
            kids = [n for n in range(1, t.n) if t.depth[n] == d]
            if not kids:
                continue
            m = max(np.float32(t.score[p] + lps[d - 1, 0]) for p in par)
            thr = np.float32(m + log_mu)
            assert all(t.score[n] >= thr for n in kids)


def test_talon_mu_one_is_a_chain_and_flat_fills_first_layer():
    rng = np.random.default_rng(4)
    # mu = 1 with distinct scores: one node per layer after the root layer
    lps, ids, Kc, _ = _talon_case(rng, 30, 6, 20, 3, 1.0)
    t = oracle.talon(lps[:, :Kc], ids[:, :Kc], 3, np.float32(0.0), 20)
    depths = t.depth[1:t.n].tolist()
    assert depths.count(1) == 3 and all(depths.count(d) == 1 for d in range(2, 7))
    # near-flat positions and mu -> 0: every child passes, the second layer
    # overflows the budget and is truncated breadth-first
    lps, ids, Kc, _ = _talon_case(rng, 30, 6, 20, 4, 1e-6, flat=True)
    t = oracle.talon(lps[:, :Kc], ids[:, :Kc], 4, np.float32(math.log(1e-6)), 20)
    assert t.n - 1 == 20
    assert set(t.depth[1:t.n].tolist()) == {1, 2}


def test_equal_scores_put_ancestors_first():
    # [DARTree] Lemma 1: on equal scores ancestors come first.  A drafter that is
    # certain at position 2 (lp = 0 for its top token) gives every depth-2 child
    # of rank 0 its parent's score; the node order must still put the parent
    # first, so the output stays topological, and DARTree's TopB(S) still equals
    # the best-first heap (beta = 0, every log-probability <= 0).
    lp = np.array([[-0.5, -1.0, -2.0, -3.0],
                   [0.0, -100.0, -100.0, -100.0],
                   [-0.25, -1.5, -2.5, -3.5]], np.float32)
    ids = np.tile(np.arange(4, dtype=np.int32), (3, 1))
    t = oracle.talon(lp, ids, 2, np.float32(math.log(0.3)), 8)
    ties = 0
    for n in range(1, t.n):
        assert t.parent[n] < n, (n, t.parent[:t.n])
        ties += int(t.score[n] == t.score[t.parent[n]])
    assert ties >= 2  # both depth-1 nodes have an equal-score child
    U = np.zeros((4, 8), np.float32)
    tree, info, _ = oracle.dartree(lp, ids, U, U, -1, 4, 0.0, 10, Mmax=11)
    assert info["topb_equals_bestfirst"]
    assert all(tree.parent[n] < n for n in range(1, tree.n))
    assert sum(int(tree.score[n] == tree.score[tree.parent[n]]) for n in range(1, tree.n)) >= 2


# --------------------------------------------------------------------------
# Tree mask
# --------------------------------------------------------------------------
def test_mask_hand_drawn_depth3():
    g = read_golden("mask_depth3.txt")
    par = np.array([int(v) for v in g["parent"][0]], np.int32)
    dep = np.array([int(v) for v in g["depth"][0]], np.int32)
    M = par.size
    t = oracle.Tree(np.zeros(M, np.int32), par, dep, np.zeros(M, np.int32), np.zeros(M, np.float32), M)
    rc, mask, pos = oracle.tree_mask(t, M, 3, pos_offset=100)
    assert rc == 0
    for n in range(M):
        want = [int(v) for v in g["row%d" % n][0]]
        got = [(int(mask[n, m // 32]) >> (m % 32)) & 1 for m in range(M)]
        assert got == want, n
    assert pos[:M].tolist() == (dep + 100).tolist()


def test_mask_invariants_and_bad_trees():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((16, 5000)) * 3).astype(np.float32)
    _, _, ids, lps = oracle.candidates(x, 40)
    t = oracle.ddtree(lps, ids, 100)
    Mmax = 101
    rc, mask, pos = oracle.tree_mask(t, Mmax, 16)
    assert rc == 0
    bits = np.unpackbits(mask.view(np.uint8), bitorder="little").reshape(Mmax, -1)[:, :Mmax]
    for n in range(t.n):
        assert bits[n].sum() == t.depth[n] + 1
        anc = set()
        a = n
        while a != -1:
            anc.add(a)
            a = t.parent[a]
        assert set(np.nonzero(bits[n])[0].tolist()) == anc
    bad = t.trimmed()
    bad.parent[5] = 5
    assert oracle.tree_mask(bad, Mmax, 16)[0] == -5
    bad = t.trimmed()
    bad.depth[7] += 1
    assert oracle.tree_mask(bad, Mmax, 16)[0] == -5
    bad = t.trimmed()
    bad.parent[3] = t.n + 2
    assert oracle.tree_mask(bad, Mmax, 16)[0] == -5


# --------------------------------------------------------------------------
# Verification
# --------------------------------------------------------------------------
def _chain_tree(tokens):
    n = len(tokens) + 1
    return oracle.Tree(np.array([-1] + list(tokens), np.int32), np.arange(-1, n - 1, dtype=np.int32),
                       np.arange(n, dtype=np.int32), np.array([-1] + [0] * (n - 1), np.int32),
                       np.zeros(n, np.float32), n)


def test_verify_greedy_chain_rule():
    V, L = 10, 4
    rng = np.random.default_rng(0)
    tokens = [3, 1, 4, 1]
    for first_bad in range(5):
        tgt = rng.standard_normal((L + 1, V)).astype(np.float32)
        for i in range(L + 1):
            want = tokens[i] if i < L else 9
            if i == first_bad:
                want = (want + 2) % V
            tgt[i, want] = 10.0
        acc, alen, nxt = oracle.verify_greedy(_chain_tree(tokens), tgt, L)
        expect_len = min(first_bad, L)
        assert alen == expect_len
        assert acc[:alen + 1].tolist() == list(range(alen + 1))
        assert nxt == int(np.argmax(tgt[alen]))


def test_verify_greedy_ties_go_to_the_smallest_token_id():
    # [Unit11] temperature section: a greedy tie goes to the smallest vocabulary
    # index.  Row 0 peaks at tokens 2 and 5 alike; the root's children carry 5
    # (rank 0) and 2 (rank 1): the walk must take token 2's child.
    V, L = 8, 3
    t = oracle.Tree(np.array([-1, 5, 2], np.int32), np.array([-1, 0, 0], np.int32), np.array([0, 1, 1], np.int32),
                    np.array([-1, 0, 1], np.int32), np.zeros(3, np.float32), 3)
    tgt = np.zeros((3, V), np.float32)
    tgt[0, [2, 5]] = 4.0
    tgt[2, 7] = 3.0
    tgt[1, 6] = 3.0
    acc, alen, nxt = oracle.verify_greedy(t, tgt, L)
    assert alen == 1 and acc[1] == 2 and nxt == 7


def test_draw_at_a_mass_boundary_takes_the_next_token():
    # The draw is an inverse CDF over half-open intervals: with two equal masses
    # a uniform of exactly 1/2 lies at the start of the second token's interval.
    # A root without children draws its token from the target row alone.
    V, L, Mmax = 4, 2, 1
    root = oracle.Tree(np.array([-1], np.int32), np.array([-1], np.int32), np.array([0], np.int32),
                       np.array([-1], np.int32), np.zeros(1, np.float32), 1)
    tgt = np.array([[1.5, 1.5, -np.inf, -np.inf]], np.float32)
    draft = np.zeros((L, V), np.float32)
    dl = np.full(L, np.log(V), np.float32)
    for u1, want in ((0.5, 1), (0.4999999, 0), (0.0, 0), (0.9999999, 1)):
        u = np.array([[0.0], [u1]], np.float32)
        for rule in ("ratio", "target_match"):
            _, alen, nxt, _ = oracle.verify_t1(root, tgt, draft, dl, u, L, Mmax, rule=rule)
            assert alen == 0 and nxt == want, (u1, rule, nxt)


def test_verify_greedy_equals_sequential_greedy_with_hash_target():
    # A deterministic "target model": the argmax after a prefix is a hash of the
    # prefix.  Tree verification must emit exactly what sequential greedy
    # decoding emits, for as long as the greedy path stays inside the tree.
    V, L = 11, 6
    rng = np.random.default_rng(12)

    def greedy_next(prefix):
        h = 7
        for t in prefix:
            h = (h * 31 + t + 1) % 1000003
        return h % V

    for trial in range(20):
        x = (rng.standard_normal((L, V)) * 1.5).astype(np.float32)
        _, _, ids, lps = oracle.candidates(x, 4)
        t = oracle.ddtree(lps, ids, 30)
        tgt = rng.standard_normal((t.n, V)).astype(np.float32)
        for n in range(t.n):
            path, a = [], n
            while a != 0:
                path.append(int(t.tok[a]))
                a = int(t.parent[a])
            tgt[n, greedy_next(tuple(reversed(path)))] = 50.0
        acc, alen, nxt = oracle.verify_greedy(t, tgt, L)
        # sequential greedy: keep decoding while the produced token is a child in the tree
        seq, node = [], 0
        while True:
            tok = greedy_next(tuple(seq))
            kids = [c for c in range(1, t.n) if t.parent[c] == node and t.tok[c] == tok]
            if not kids:
                break
            seq.append(tok)
            node = kids[0]
        assert alen == len(seq)
        assert nxt == greedy_next(tuple(seq))
        assert 1 <= alen + 1 <= L + 1


def test_worked_example_scalar_rule():
    g = read_golden("three_token_example.txt")
    q = np.array([float(v) for v in g["q"][0]])
    p = np.array([float(v) for v in g["p"][0]])
    _, _, a, r = oracle.spec_scalar(p, q, 0.5, 0.5, 0.5)
    assert np.allclose(a, [float(v) for v in g["accept"][0]], atol=1e-12)
    assert np.allclose(r, [float(v) for v in g["residual"][0]], atol=1e-12)
    assert abs(float(np.sum(q * (1 - a))) - float(g["rejected_mass"][0][0])) < 1e-12
    # lossless identity min(p, q) + R * r = p
    R = float(np.sum(np.maximum(q - p, 0)))
    assert np.allclose(np.minimum(p, q) + R * r, p, atol=1e-12)


def test_worked_example_frequencies_within_3_sigma():
    g = read_golden("three_token_example.txt")
    q = np.array([float(v) for v in g["q"][0]])
    p = np.array([float(v) for v in g["output"][0]])
    n = 1_000_000
    u = np.random.default_rng(2024).random((n, 3))
    counts = oracle.spec_scalar_trials(p, q, u)
    freq = counts / n
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(freq - p) <= 3 * sigma), (freq, p)


def test_tree_t1_on_worked_example_frequencies_and_fixed_point_residual():
    # The tree walk's T=1 arithmetic (exp_canon ratios, 2^32 fixed-point
    # residual, inverse-CDF draw) on the worked example through a one-child
    # tree: drafted token x ~ q, accepted or replaced; the emitted token must be
    # distributed as p.
    g = read_golden("three_token_example.txt")
    q = np.array([float(v) for v in g["q"][0]])
    p = np.array([float(v) for v in g["p"][0]])
    lq = np.log(q).astype(np.float32)[None, :]
    lp = np.log(p).astype(np.float32)
    draft_lse = np.zeros(1, np.float32)
    rng = np.random.default_rng(77)
    n = 100_000
    counts = np.zeros(3, np.int64)
    for _ in range(n):
        ud, ua, ur = rng.random(3)
        x = int(np.searchsorted(np.cumsum(q), ud, side="right"))
        t = _chain_tree([x])
        t.rank[1] = 0
        tgt = np.stack([lp, lp])  # row 1 unused unless accepted (then only the bonus draw)
        u = np.array([[0.0, ua], [ur, 0.5]], np.float32)
        acc, alen, nxt, _ = oracle.verify_t1(t, tgt, lq, draft_lse, u, 1, 2, lse_in=np.zeros(2, np.float32))
        counts[x if alen == 1 else nxt] += 1
    freq = counts / n
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(freq - p) <= 3 * sigma), (freq, p)
    # after rejecting C the residual gives A:B = 1:3 exactly up to 2^-32 fixed point
    t = _chain_tree([2])
    t.rank[1] = 0
    got = []
    for ur in np.linspace(0.0005, 0.9995, 1000):
        u = np.array([[0.0, 0.9999], [ur, 0.5]], np.float32)
        acc, alen, nxt, _ = oracle.verify_t1(t, np.stack([lp, lp]), lq, draft_lse, u, 1, 2,
                                              lse_in=np.zeros(2, np.float32))
        assert alen == 0
        got.append(nxt)
    assert got.count(2) == 0
    assert got.count(0) == 250 and got.count(1) == 750


def test_t1_edge_cases_r_zero_and_p_zero():
    # p = q: R = 0, every draft is accepted (ratio exp(0) = 1 > u)
    lq = np.log(np.array([[0.3, 0.7]])).astype(np.float32)
    t = _chain_tree([1])
    t.rank[1] = 0
    for ua in (0.0, 0.5, 0.999999):
        u = np.array([[0.0, ua], [0.3, 0.3]], np.float32)
        _, alen, _, _ = oracle.verify_t1(t, np.stack([lq[0], lq[0]]), lq, np.zeros(1, np.float32), u, 1, 2,
                                         lse_in=np.zeros(2, np.float32))
        assert alen == 1
    # p(x) = 0 < q(x): always rejected, and x never re-emitted
    tgt = np.array([0.0, -np.inf], np.float32)
    for ua in (0.0, 0.5):
        u = np.array([[0.0, ua], [0.9, 0.3]], np.float32)
        _, alen, nxt, _ = oracle.verify_t1(t, np.stack([tgt, tgt]), lq, np.zeros(1, np.float32), u, 1, 2,
                                           lse_in=np.zeros(2, np.float32))
        assert alen == 0 and nxt == 0


def test_t1_rejection_with_an_empty_residual_draws_from_p():
    # A rejected child whose residual is empty: the replacement comes from p.
    # Target and drafter rows are the same logits, but the drafter's supplied
    # normaliser sits 0.001 below the true one, so every drafter mass is at
    # least the target's (the residual [p - q]_+ is empty) while the child's
    # ratio is exp(-0.001) ~ 0.999 < u.  Row: two equal masses, so a draw
    # uniform of 1/2 lies at the start of the second token's interval.
    V = 6
    row = np.full(V, -30.0, np.float32)
    row[[0, 4]] = 1.5
    lse = np.float32(np.logaddexp.reduce(row.astype(np.float64)))
    t = _chain_tree([0])
    t.rank[1] = 0
    u = np.array([[0.0, 0.9999], [0.5, 0.5]], np.float32)
    acc, alen, nxt, _ = oracle.verify_t1(t, np.stack([row, row]), row[None, :], np.array([lse - 0.001], np.float32),
                                         u, 1, 2)
    assert alen == 0 and nxt == 4
