"""End-to-end selection check -- TEST INFRASTRUCTURE (part of the oracle).

When the GPU computes stage 1 itself from raw logits, its candidate tables
carry the same ids as the oracle's (bit-exact) and log-probs within the stated
1e-5 of the oracle's.  Every tree score is a path sum of such log-probs, so a
selection can legitimately differ from the oracle's where two candidates' path
scores lie within the error those sums can accumulate.  This module decides,
for a tree selected elsewhere ("got") and the oracle's own tree ("want"),
whether every difference is such a near-tie, and counts them.

Tolerance of one node's score (derived from the per-log-prob contract).  A
node at depth d has the path score S_d = fl(fl(S_{d-1} + t_d) + beta) with
t_d the edge term (the log-prob, plus the DARTree / heap edge term and minus
the normaliser where used); the oracle computes the same sums from its own
table.  With |t_g - t_o| <= eps_t per edge (eps_t = eps_lp, plus eps_z for a
normaliser computed elsewhere) and fp32 round-to-nearest (relative error
u = 2^-24 per operation on either side), the two sums differ by at most

    tau(d) = sum_{j=1..d} [ eps_t + 2^-23 * (|t_j| + |S_{j-1} + t_j| + |S_j|) ]

(each rounding contributes at most u times the value on each side, the
values on the two sides agreeing to within tau).  With eps_lp = 1e-5 a
depth-16 path may move by 1.6e-4 plus rounding: the near-tie window of a
tree is wider than the per-log-prob 1e-5 and grows with depth.

A selection difference is a near-tie when the node that differs first on its
path (its parent is in both trees) has an oracle score within
tau(node) + tau(other) of a cut the selection makes at that depth, tau(other)
the largest tolerance among the cut's own node and the differing nodes (a
node a that one tree keeps and the other drops was exchanged for some node b
on the other side of the cut, and s(b) - s(a) <= tau(a) + tau(b)):

  - the last selected score (the B-th: DDTree, heap, DARTree's final Top-B);
  - the lowest kept score among the want tree's nodes of that depth (a
    DARTree width cut, a TALON truncation);
  - TALON's gate m_d + log mu (m_d the best score of the depth).

Descendants of such a node differ as a consequence and are counted apart.
DARTree and TALON select layer by layer from the children of the previous
layer, so once a layer differs, the next layer's pool differs too and may
push out a node whose parent both trees share: below the first layer that
differs, differences are counted as consequences in those two modes.  In the
best-first modes (DDTree, heap) every differing node at every depth must be a
near-tie of the last selected score.
Nodes present in both trees but listed in another order must be within the
sum of their tolerances of each other.  Passages: the score definitions of
[DDTree] section 3.3 (log-domain path sums), [DARTree] Algorithm 1 and the
equation of s_beta, [TALON] key designs 1-2 (the gate and the truncation).
"""
import numpy as np

TWO_M23 = 2.0 ** -23


def _order_by_depth(tree):
    n = tree.n
    return sorted(range(1, n), key=lambda i: int(tree.depth[i]))


def path_scores(tree, cand_lp, mode, E=None, znorm=None, beta=0.0, root_term=False):
    """Oracle-arithmetic score of every node of `tree` from the table cand_lp
    [L, K] (fp32, one rounding per operation as the oracle does it), with the
    per-node tolerance terms.  tree.rank holds each node's candidate rank.
    mode: "ddtree", "talon", "dartree" or "heap"; E [L, K, K]: edge terms
    (row 0 of position 0: the root); znorm [L, K]: log-normalisers;
    root_term: DARTree adds the edge term (and normaliser) at depth 1.
    Returns (scores, paths, parts): scores float32 [n]; paths: tuple of ranks
    per node; parts: per node the list of (|t|, |S_prev + t|, |S|) per level."""
    lp = np.asarray(cand_lp, np.float32)
    n = tree.n
    f = np.float32
    s = np.zeros(n, np.float32)
    paths = [()] * n
    parts = [[] for _ in range(n)]
    beta32 = f(beta)
    for i in _order_by_depth(tree):
        p = int(tree.parent[i])
        d = int(tree.depth[i])
        r = int(tree.rank[i])
        if p < 0 or p >= n or d < 1 or int(tree.depth[p]) != d - 1:
            raise ValueError("node %d: not a tree (parent %d, depth %d)" % (i, p, d))
        prow = 0 if d == 1 else int(tree.rank[p])
        t = lp[d - 1, r]
        if mode == "dartree":
            if E is not None and (d > 1 or root_term):
                t = f(t + E[d - 1, prow, r])
                if znorm is not None:
                    t = f(t - znorm[d - 1, prow])
            mid = f(s[p] + t)
            s[i] = f(mid + beta32)
        elif mode == "heap":
            if E is not None:
                t = f(t + E[d - 1, prow, r])
            if znorm is not None:
                t = f(t - znorm[d - 1, prow])
            mid = f(s[p] + t)
            s[i] = mid
        else:
            mid = f(s[p] + t)
            s[i] = mid
        paths[i] = paths[p] + (r,)
        parts[i] = parts[p] + [(abs(float(t)), abs(float(mid)), abs(float(s[i])))]
    return s, paths, parts


def _tau(parts, eps_t):
    return sum(eps_t + TWO_M23 * (a + b + c) for a, b, c in parts) * (1.0 + 2.0 ** -10)


def selection_check(got, want, cand_lp, mode, eps_lp=1e-5, eps_z=0.0, E=None, znorm=None, beta=0.0,
                    root_term=False, log_mu=None, got_scores=None):
    """Compare tree `got` (selected from another stage-1 table of the same
    ids) with the oracle's tree `want` (selected from cand_lp).  Both trees
    carry candidate ranks.  got_scores: got's own scores (checked against the
    oracle rescoring within tau).  Returns a dict:
      differing     -- nodes (paths) in exactly one tree
      near_ties     -- differing nodes whose parent is in both trees, each
                       within its tolerance of a cut (see the module text)
      consequences  -- differing nodes below a differing parent
      mismatches    -- differing nodes whose parent is in both trees and that
                       are beyond every cut's tolerance (must be empty)
      order_swaps   -- pairs in both trees listed in opposite orders
      order_mismatches -- such pairs farther apart than their tolerances
      score_err_max, score_err_viol -- |got score - oracle rescoring| and the
                       nodes where it exceeds tau
      tau_max       -- the largest node tolerance seen."""
    eps_t = eps_lp + eps_z
    sw, pw, qw = path_scores(want, cand_lp, mode, E, znorm, beta, root_term)
    want_scores = np.asarray(want.score[:want.n], np.float32)
    bad = np.nonzero(sw[1:].view(np.uint32) != want_scores[1:].view(np.uint32))[0]
    if bad.size:
        raise AssertionError("the rescoring does not reproduce the oracle's own scores at nodes %s" % (bad[:5] + 1))
    sg, pg, qg = path_scores(got, cand_lp, mode, E, znorm, beta, root_term)
    tw = {pw[i]: (float(sw[i]), _tau(qw[i], eps_t), i) for i in range(1, want.n)}
    tg = {pg[i]: (float(sg[i]), _tau(qg[i], eps_t), i) for i in range(1, got.n)}

    # cuts of the want tree
    cuts = {}
    if want.n > 1:
        last = min(range(1, want.n), key=lambda i: (float(sw[i]), -i))
        glob = (float(sw[last]), tw[pw[last]][1])
    else:
        glob = None
    by_depth = {}
    for i in range(1, want.n):
        by_depth.setdefault(int(want.depth[i]), []).append(i)
    for d, nodes in by_depth.items():
        lo = min(nodes, key=lambda i: float(sw[i]))
        hi = max(nodes, key=lambda i: float(sw[i]))
        c = [(float(sw[lo]), tw[pw[lo]][1])]
        if log_mu is not None and d > 1:
            gate = float(np.float32(sw[hi] + np.float32(log_mu)))
            c.append((gate, tw[pw[hi]][1] + TWO_M23 * abs(gate)))
        cuts[d] = c

    diff = set(tw) ^ set(tg)
    layerwise = mode in ("dartree", "talon")
    first = min((len(p) for p in diff), default=0)
    tau_diff = {}
    for path in diff:
        d = len(path)
        tau_diff[d] = max(tau_diff.get(d, 0.0), (tw.get(path) or tg.get(path))[1])
    tau_diff_all = max(tau_diff.values(), default=0.0)
    near, cons, mism = [], [], []
    for path in sorted(diff, key=len):
        parent = path[:-1]
        if (parent and parent in diff) or (layerwise and len(path) > first):
            cons.append(path)
            continue
        s, tau, _ = tw.get(path) or tg.get(path)
        d = len(path)
        cand = [(c, max(tc, tau_diff[d])) for c, tc in cuts.get(d, [])]
        if glob is not None:
            cand.append((glob[0], max(glob[1], tau_diff_all)))
        gap = min((abs(s - c) - tau - tc for c, tc in cand), default=float("inf"))
        (near if gap <= 0.0 else mism).append((path, s, gap))

    # order of the common nodes
    common = [p for p in (pg[i] for i in range(1, got.n)) if p in tw]
    pos_w = np.array([tw[p][2] for p in common])
    swaps = order_bad = 0
    if len(common) > 1:
        sc = np.array([tw[p][0] for p in common])
        ta = np.array([tw[p][1] for p in common])
        inv = pos_w[:, None] > pos_w[None, :]
        inv = np.triu(inv, 1)
        swaps = int(inv.sum())
        if swaps:
            far = np.abs(sc[:, None] - sc[None, :]) > ta[:, None] + ta[None, :]
            order_bad = int((inv & far).sum())

    err_max, err_viol = 0.0, 0
    if got_scores is not None:
        gs = np.asarray(got_scores[:got.n], np.float64)
        for i in range(1, got.n):
            e = abs(gs[i] - float(sg[i]))
            err_max = max(err_max, e)
            if e > _tau(qg[i], eps_t):
                err_viol += 1
    tau_max = max([v[1] for v in tw.values()] + [v[1] for v in tg.values()] + [0.0])
    return dict(differing=len(diff), near_ties=len(near), consequences=len(cons), mismatches=mism,
                order_swaps=swaps, order_mismatches=order_bad, score_err_max=err_max, score_err_viol=err_viol,
                tau_max=tau_max, near_tie_detail=near)
