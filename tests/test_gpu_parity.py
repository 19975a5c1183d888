"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Inputs only flow from the oracle to the GPU, never back:
  - stage 1 runs on both sides from the same raw logits: ids bit-exact,
    normalisers and log-probs within 1e-5;
  - selection, mask and walk are bit-exact when the GPU entry points are fed
    the oracle's fp32 candidate tables, trees and target normalisers (the ABI
    accepts caller-supplied tables, trees and normalisers);
  - end to end (the GPU computing everything itself from raw logits), any tree
    difference must come from a near-tie (a score within 1e-5 of the last
    selected one) and is counted; walks must agree.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from speculative_decoding_draft_bf16_gb300 import workloads as wk

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def gen_logits(batch, L, V, dtype, scale=3.0, p_spike=0.7, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((batch, L, V), generator=g) * scale
    if p_spike > 0:
        has = torch.rand((batch, L), generator=g) < p_spike
        tok = torch.randint(0, V, (batch, L), generator=g)
        bi, li = torch.nonzero(has, as_tuple=True)
        x[bi, li, tok[bi, li]] += 8.0
    return x.to(torch.bfloat16) if dtype == "bf16" else x


def f32(t):
    return t.float().cpu().numpy()


def gpu_tree(tree, b):
    n = int(tree.n_nodes[b])
    return oracle.Tree(tree.node_tok[b].cpu().numpy()[:n].copy(), tree.parent[b].cpu().numpy()[:n].copy(),
                       tree.depth[b].cpu().numpy()[:n].copy(), tree.rank[b].cpu().numpy()[:n].copy(),
                       tree.score[b].cpu().numpy()[:n].copy(), n)


def assert_same_tree(g, o, what=""):
    assert g.n == o.n, (what, g.n, o.n)
    n = g.n
    for f in ("tok", "parent", "depth", "rank"):
        a, b = getattr(g, f)[:n], getattr(o, f)[:n]
        assert np.array_equal(a, b), (what, f, np.nonzero(a != b)[0][:10])
    assert np.array_equal(g.score[:n].view(np.uint32), o.score[:n].view(np.uint32)), what


# End to end, the GPU's own stage-1 tables carry the oracle's ids and log-probs
# within TOL, and every tree score is a path sum of them: a selection may differ
# from the oracle's only by near-ties, within the per-node tolerance
# oracle.selection_check derives from TOL (it grows with depth, up to about
# 1.6e-4 plus rounding at depth 16).  Each end-to-end case states how many
# near-tie nodes it accepts per request: one exchange across a cut is two
# nodes (one kept by each side).  Spiky rows have scores far apart, and
# allow one exchange; rows with massive ties allow more (stated per case).
NEAR_TIES_PER_REQUEST = 2
NEAR_TIE_TALLY = {"requests": 0, "near_ties": 0, "consequences": 0, "order_swaps": 0, "score_err_max": 0.0}


def check_end_to_end(g, o, lps, mode, max_near_ties=NEAR_TIES_PER_REQUEST, what="", **kw):
    """GPU tree g (from its own stage 1) against the oracle tree o (from the
    oracle's table lps): every difference a near-tie, the count within
    max_near_ties, every GPU score within its tolerance of the oracle's
    arithmetic on the same path."""
    rep = oracle.selection_check(g, o, lps, mode, eps_lp=TOL, got_scores=g.score, **kw)
    assert rep["mismatches"] == [], ("selection differs beyond a near-tie", what, rep["mismatches"][:3])
    assert rep["order_mismatches"] == 0, ("node order differs beyond a near-tie", what)
    assert rep["score_err_viol"] == 0, ("a score beyond its tolerance", what, rep["score_err_max"])
    assert rep["near_ties"] <= max_near_ties, ("more near-ties than the case allows", what, rep["near_ties"])
    NEAR_TIE_TALLY["requests"] += 1
    for k in ("near_ties", "consequences", "order_swaps"):
        NEAR_TIE_TALLY[k] += rep[k]
    NEAR_TIE_TALLY["score_err_max"] = max(NEAR_TIE_TALLY["score_err_max"], rep["score_err_max"])
    print("end to end %s: near-ties %d, consequences %d, order swaps %d, max score error %.2e (tolerance up to %.2e)"
          % (what, rep["near_ties"], rep["consequences"], rep["order_swaps"], rep["score_err_max"], rep["tau_max"]))
    return rep


def oracle_tables(x_b, Kc):
    """Oracle stage 1 for one request: (lse32 [L], ids [L, Kc], lps [L, Kc])."""
    _, l32, ids, lps = oracle.candidates(f32(x_b), Kc)
    return l32, ids, lps


def upload_tables(tree, b, l32, ids, lps):
    tree.lse[b].copy_(torch.from_numpy(l32))
    tree.cand_id[b].copy_(torch.from_numpy(ids))
    tree.cand_lp[b].copy_(torch.from_numpy(lps))


def upload_tree(tree, b, t):
    n = t.n
    tree.node_tok[b, :n] = torch.from_numpy(t.tok[:n])
    tree.parent[b, :n] = torch.from_numpy(t.parent[:n])
    tree.depth[b, :n] = torch.from_numpy(t.depth[:n])
    tree.rank[b, :n] = torch.from_numpy(t.rank[:n])
    tree.score[b, :n] = torch.from_numpy(t.score[:n])
    tree.n_nodes[b] = n


def row_lse(rows):
    """Oracle normaliser (double, rounded to fp32) of each row of [n, V]."""
    _, l32, _, _ = oracle.candidates(rows, 1)
    return l32


# ---------------------------------------------------------------------------
# Stage 1: GPU and oracle from the same raw logits
# ---------------------------------------------------------------------------
CAND_CASES = [
    (1, 4, 32, "f32", 4, 2.0, 0.0),          # tiny greedy shape: one CTA, fp32
    (2, 3, 1000, "bf16", 17, 3.0, 0.7),      # ragged vocabulary, several chunks
    (3, 2, 1001, "bf16", 64, 3.0, 0.7),      # odd V: rows not 16-byte aligned (head/tail loads)
    (2, 2, 5000, "f32", 100, 3.0, 0.7),      # fp32: window + two low-bit radix rounds
    (1, 16, 151936, "bf16", 256, 3.0, 0.7),  # single request at Qwen3 vocabulary (16-CTA clusters)
    (2, 4, 151936, "bf16", 1024, 3.0, 0.7),  # largest candidate list
    (1, 2, 151936, "f32", 64, 3.0, 0.7),
    (20, 16, 151936, "bf16", 60, 3.0, 0.5),  # many rows: persistent clusters prefetching their next row
    (8, 16, 151936, "bf16", 1024, 3.0, 0.7),  # many rows, largest list: sorted ranking
    (6, 16, 151936, "f32", 256, 3.0, 0.7),    # many fp32 rows
    (4, 16, 300000, "f32", 64, 3.0, 0.7),     # long fp32 rows: > 32 vectors per maximum slot
    (4, 16, 10001, "bf16", 32, 3.0, 0.7),     # many rows, odd V: rows not 16-byte aligned
    (4, 16, 10001, "bf16", 200, 3.0, 0.7),    # long lists (per-vector words), rows not 16-byte aligned
    (5, 16, 20000, "bf16", 129, 3.0, 0.7),    # the shortest list on the per-vector words: counting rank
    (4, 16, 300000, "bf16", 256, 3.0, 0.7),   # long bf16 rows: two vectors per word, unordered ranking
]


@pytest.mark.parametrize("batch,L,V,dtype,Kc,scale,p_spike", CAND_CASES)
def test_candidates_parity(batch, L, V, dtype, Kc, scale, p_spike):
    x = gen_logits(batch, L, V, dtype, scale, p_spike, seed=V + Kc)
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype=dtype, K=Kc, B=Kc)
    tree = dtree.TreeBuffers.for_params(p)
    dtree.candidates(p, x.cuda(), tree)
    torch.cuda.synchronize()
    rows = list(range(batch * L)) if batch * L <= 64 else list(range(0, batch * L, 7))
    xs = f32(x).reshape(batch * L, V)[rows]
    lse64, _, ids, lps = oracle.candidates(xs, Kc)
    g_ids = tree.cand_id.cpu().numpy().reshape(batch * L, Kc)[rows]
    g_lp = tree.cand_lp.cpu().numpy().reshape(batch * L, Kc)[rows]
    g_lse = tree.lse.cpu().numpy().reshape(batch * L)[rows]
    assert np.array_equal(g_ids, ids)
    assert np.max(np.abs(g_lse - lse64)) < TOL
    assert np.max(np.abs(g_lp - lps)) < TOL
    # each lp is the logit minus the row's normaliser, one fp32 subtraction
    want = (np.take_along_axis(xs, g_ids, 1) - g_lse[:, None]).astype(np.float32)
    assert np.array_equal(g_lp.view(np.uint32), want.view(np.uint32))
    assert int(tree.status.abs().sum()) == 0


@pytest.mark.parametrize("batch,L,V,dtype,Kc", [(1, 16, 151936, "bf16", 256), (2, 3, 1001, "bf16", 64),
                                                 (1, 2, 5000, "f32", 100)])
def test_stage1_ceiling_reads_every_element(batch, L, V, dtype, Kc):
    # the measurement kernel with the cluster stage-1 launch: the maximum of each
    # row's chunk maxima is the row maximum (every element was read)
    x = gen_logits(batch, L, V, dtype, 3.0, 0.7, seed=V).cuda()
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype=dtype, K=Kc, B=Kc)
    kind, S = dtree.stage1_plan(p)
    assert kind == "cluster"
    out = torch.full((batch * L, S), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dtree.stage1_ceiling(p, x, out, st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    assert torch.equal(out.max(dim=1).values, x.float().reshape(batch * L, V).max(dim=1).values)


def test_candidates_edge_rows():
    # all-equal row (smallest ids win), one outlier far above the rest (the
    # 256-step key window holds too few keys: full radix path), -inf entries,
    # a row with only two finite logits
    V, Kc = 20000, 50
    x = torch.randn((4, V)) * 2
    x[0] = 1.5
    x[1, 123] = 1e30
    x[2, ::3] = -float("inf")
    x[3, :] = -float("inf")
    x[3, 7] = 0.0
    x[3, 19999] = 0.0
    for dtype in ("bf16", "f32"):
        xx = x.to(torch.bfloat16) if dtype == "bf16" else x.clone()
        p = dtree.Params(mode="ddtree", batch=1, L=4, V=V, dtype=dtype, K=Kc, B=Kc)
        tree = dtree.TreeBuffers.for_params(p)
        dtree.candidates(p, xx.reshape(1, 4, V).contiguous().cuda(), tree)
        torch.cuda.synchronize()
        lse64, _, ids, lps = oracle.candidates(f32(xx), Kc)
        assert np.array_equal(tree.cand_id[0].cpu().numpy(), ids)
        assert np.max(np.abs(tree.lse[0].cpu().numpy() - lse64)) < TOL
        assert tree.cand_id[0, 3, :2].cpu().tolist() == [7, 19999]
        assert abs(float(tree.lse[0, 3]) - math.log(2.0)) < TOL


@pytest.mark.parametrize("batch,Kc", [(6, 40), (16, 40), (6, 200)])
def test_candidates_edge_rows_among_many(batch, Kc):
    # many rows, so that CTAs or clusters run through several rows in turn;
    # edge rows (equal logits, an outlier, -inf runs) between Gaussian rows
    # switch between the candidate path and the exact fallback from one row to
    # the next (Kc = 200: on the per-vector words, whose bound can list every
    # vector of a row and overflow into several staged rounds)
    L, V = 16, 20000
    g = torch.Generator().manual_seed(99)
    x = torch.randn((batch * L, V), generator=g) * 2
    for r in range(0, batch * L, 5):
        kind = (r // 5) % 4
        if kind == 0:
            x[r] = 0.75
        elif kind == 1:
            x[r, (r * 37) % V] = 1e30
        elif kind == 2:
            x[r, r % 3::3] = -float("inf")
        else:
            x[r] = -float("inf")
            x[r, r % V] = 1.0
    for dtype in ("bf16", "f32"):
        xx = x.to(torch.bfloat16) if dtype == "bf16" else x.clone()
        p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype=dtype, K=Kc, B=Kc)
        tree = dtree.TreeBuffers.for_params(p)
        dtree.candidates(p, xx.reshape(batch, L, V).contiguous().cuda(), tree)
        torch.cuda.synchronize()
        xs = f32(xx)
        lse64, _, ids, lps = oracle.candidates(xs, Kc)
        g_ids = tree.cand_id.cpu().numpy().reshape(batch * L, Kc)
        g_lse = tree.lse.cpu().numpy().reshape(batch * L)
        assert np.array_equal(g_ids, ids), dtype  # -inf ties too: smallest ids first
        assert np.max(np.abs(g_lse - lse64)) < TOL, dtype
        g_lp = tree.cand_lp.cpu().numpy().reshape(batch * L, Kc)
        finite = np.isfinite(lps)
        assert np.array_equal(g_lp[~finite], lps[~finite]), dtype
        assert np.max(np.abs(g_lp[finite] - lps[finite])) < TOL, dtype
        assert int(tree.status.abs().sum()) == 0


# ---------------------------------------------------------------------------
# DDTree selection
# ---------------------------------------------------------------------------
DD_CASES = [
    (1, 4, 32, "f32", 4, 8, 2.0, 0.0),
    (3, 5, 700, "bf16", 6, 40, 3.0, 0.7),
    (2, 8, 3000, "bf16", 32, 200, 1.0, 0.3),   # flat rows: deep, wide trees and many ties
    (2, 16, 5000, "bf16", 64, 64, 3.0, 0.7),
    (1, 16, 151936, "bf16", 128, 128, 3.0, 0.7),
    (2, 3, 500, "bf16", 3, 39, 3.0, 0.0),      # B = |S_K|: the whole prefix set
    (2, 2, 400, "bf16", 8, 1024, 3.0, 0.7),    # B far above |S_K|
    (1, 6, 4000, "bf16", 256, 1024, 0.3, 0.0),  # largest budget, many candidates per depth
    (2, 16, 2000, "bf16", 16, 300, 0.05, 0.0),  # nearly uniform rows: massive score ties
    (1, 4, 3000, "bf16", 512, 600, 0.3, 0.0),   # more depth-1 nodes than threads: parents re-sorted
]


def ddtree_case(batch, L, V, dtype, K, B, scale, p_spike, seed):
    """Returns (GPU-selected tree buffers fed the oracle's tables, oracle trees, logits)."""
    x = gen_logits(batch, L, V, dtype, scale, p_spike, seed=seed)
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype=dtype, K=K, B=B)
    tree = dtree.TreeBuffers.for_params(p)
    otrees, tables = [], []
    for b in range(batch):
        l32, ids, lps = oracle_tables(x[b], K)
        upload_tables(tree, b, l32, ids, lps)
        otrees.append(oracle.ddtree(lps, ids, B).trimmed())
        tables.append(lps)
    dtree.select(p, tree)
    torch.cuda.synchronize()
    for b in range(batch):
        assert_same_tree(gpu_tree(tree, b), otrees[b], "b=%d" % b)
    return tree, otrees, x, p, tables


@pytest.mark.parametrize("batch,L,V,dtype,K,B,scale,p_spike", DD_CASES)
def test_ddtree_parity(batch, L, V, dtype, K, B, scale, p_spike):
    _, otrees, x, p, tables = ddtree_case(batch, L, V, dtype, K, B, scale, p_spike, seed=K * 7 + B)
    # end to end: the GPU alone from raw logits
    tree = dtree.TreeBuffers.for_params(p)
    dtree.build_tree(p, x.cuda(), tree)
    torch.cuda.synchronize()
    # flat rows (scale <= 1) pack many exactly tied scores at the cut, whose
    # order a rounding difference can flip: up to B/16 near-tie nodes there
    allow = NEAR_TIES_PER_REQUEST if scale > 1.0 else max(NEAR_TIES_PER_REQUEST, B // 16)
    for b in range(batch):
        check_end_to_end(gpu_tree(tree, b), otrees[b], tables[b], "ddtree", allow, "ddtree %s b=%d" % (
            (batch, L, V, dtype, K, B, scale), b))


def test_ddtree_single_request_full_size_all_budgets():
    for B in (64, 128, 256):
        wl = wk.single_request(B)
        x, _ = wk.draft_logits(wl)
        p = dtree.Params(mode="ddtree", batch=1, L=16, V=wl.V, dtype="bf16", K=B, B=B)
        tree = dtree.TreeBuffers.for_params(p)
        l32, ids, lps = oracle_tables(x[0], B)
        upload_tables(tree, 0, l32, ids, lps)
        o = oracle.ddtree(lps, ids, B).trimmed()
        dtree.select(p, tree)
        torch.cuda.synchronize()
        assert_same_tree(gpu_tree(tree, 0), o, "B=%d" % B)
        tree2 = dtree.TreeBuffers.for_params(p)
        dtree.build_tree(p, x.cuda(), tree2)
        torch.cuda.synchronize()
        check_end_to_end(gpu_tree(tree2, 0), o, lps, "ddtree", what="single request B=%d" % B)


# ---------------------------------------------------------------------------
# Tree mask (oracle trees fed to the GPU)
# ---------------------------------------------------------------------------
def tree_from_arrays(parent, depth, tok=None, L=3, Mmax=None):
    M = len(parent)
    Mmax = Mmax or M
    t = dtree.TreeBuffers(1, L, 1, Mmax)
    t.parent[0, :M] = torch.tensor(parent, dtype=torch.int32)
    t.depth[0, :M] = torch.tensor(depth, dtype=torch.int32)
    if tok is not None:
        t.node_tok[0, :M] = torch.tensor(tok, dtype=torch.int32)
    t.n_nodes[0] = M
    return t


def test_mask_hand_drawn_depth3_on_gpu():
    from conftest import read_golden
    g = read_golden("mask_depth3.txt")
    par = [int(v) for v in g["parent"][0]]
    dep = [int(v) for v in g["depth"][0]]
    t = tree_from_arrays(par, dep, L=3, Mmax=40)
    mask, pos = dtree.alloc_mask(t)
    dtree.tree_mask(t, mask, pos, pos_offset=7)
    torch.cuda.synchronize()
    m = mask[0].cpu().numpy().view(np.uint32)
    for n in range(len(par)):
        want = [int(v) for v in g["row%d" % n][0]]
        got = [(int(m[n, k // 32]) >> (k % 32)) & 1 for k in range(len(par))]
        assert got == want
        assert np.all(m[n, 1:] == 0)
    assert pos[0, :len(par)].cpu().tolist() == [d + 7 for d in dep]
    assert int(t.status[0]) == 0


@pytest.mark.parametrize("case", [1, 3, 7, 8])
def test_mask_parity_on_oracle_trees(case):
    batch, L, V, dtype, K, B, scale, p_spike = DD_CASES[case]
    tree, otrees, _, _, _ = ddtree_case(batch, L, V, dtype, K, B, scale, p_spike, seed=11)
    t2 = dtree.TreeBuffers(batch, L, K, B + 1)
    for b in range(batch):
        upload_tree(t2, b, otrees[b])
    mask, pos = dtree.alloc_mask(t2)
    dtree.tree_mask(t2, mask, pos, pos_offset=3)
    torch.cuda.synchronize()
    for b in range(batch):
        rc, om, opos = oracle.tree_mask(otrees[b], B + 1, L, pos_offset=3)
        assert rc == 0
        n = otrees[b].n
        assert np.array_equal(mask[b].cpu().numpy().view(np.uint32)[:n], om[:n])
        assert np.array_equal(pos[b, :n].cpu().numpy(), opos[:n])
    assert int(t2.status.abs().sum()) == 0


def test_mask_and_verify_flag_bad_trees():
    bad_cases = [
        ([-1, 0, 5], [0, 1, 2]),     # parent out of range
        ([-1, 0, 2], [0, 1, 2]),     # self-parent
        ([-1, 0, 1], [0, 1, 3]),     # depth jump
        ([0, 0, 1], [0, 1, 2]),      # root with a parent
    ]
    for par, dep in bad_cases:
        t = tree_from_arrays(par, dep, tok=[-1, 1, 2], L=3, Mmax=8)
        mask, pos = dtree.alloc_mask(t)
        mask.fill_(-1)
        dtree.tree_mask(t, mask, pos)
        tgt = torch.randn((1, 8, 64), device="cuda")
        out = dtree.verify(t, tgt)
        torch.cuda.synchronize()
        assert int(t.status[0]) & dtree.DT_DEV_BAD_TREE
        assert torch.all(mask == -1)  # nothing written
        assert int(out[1][0]) == 0 and int(out[2][0]) == -1


# ---------------------------------------------------------------------------
# Verification (oracle trees, oracle normalisers fed to the GPU)
# ---------------------------------------------------------------------------
def verify_tree_buffers(otrees, L, Kc, Mmax, lse_rows=None):
    t = dtree.TreeBuffers(len(otrees), L, Kc, Mmax)
    for b, o in enumerate(otrees):
        upload_tree(t, b, o)
        if lse_rows is not None:
            t.lse[b].copy_(torch.from_numpy(lse_rows[b]))
    return t


def test_verify_greedy_single_request_full_size():
    wl = wk.single_request(256)
    x, spikes = wk.draft_logits(wl)
    l32, ids, lps = oracle_tables(x[0], 256)
    o = oracle.ddtree(lps, ids, 256).trimmed()
    depth = np.zeros((1, wl.max_nodes), np.int32)
    depth[0, :o.n] = o.depth
    tgt = wk.target_logits(wl, depth, [o.n], spikes)
    t = verify_tree_buffers([o], 16, 256, wl.max_nodes)
    out = dtree.verify(t, tgt.cuda())
    torch.cuda.synchronize()
    acc, alen, nxt = oracle.verify_greedy(o, f32(tgt[0]), 16)
    assert out[0][0].cpu().tolist() == acc.tolist()
    assert int(out[1][0]) == alen and int(out[2][0]) == nxt


def stress_targets(t, V, seed):
    """Target rows whose argmax is the token of the node's rank-0 child, so
    the greedy walk goes as deep as the tree."""
    g = torch.Generator().manual_seed(seed)
    tgt = torch.randn((t.n, V), generator=g) * 3
    for n in range(t.n):
        kids = [c for c in range(1, t.n) if t.parent[c] == n]
        if kids:
            c = min(kids, key=lambda c: t.rank[c])
            tgt[n, t.tok[c]] = 40.0
    return tgt


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_greedy_deep_walks(dtype):
    batch, L, V, K, B = 3, 12, 3000, 8, 60
    x = gen_logits(batch, L, V, dtype, 0.5, 0.9, seed=5)
    otrees = [oracle.ddtree(*oracle_tables(x[b], K)[2:0:-1], B).trimmed() for b in range(batch)]
    tg = torch.zeros((batch, B + 1, V))
    for b in range(batch):
        tg[b, :otrees[b].n] = stress_targets(otrees[b], V, seed=b)
    tg = tg.to(torch.bfloat16) if dtype == "bf16" else tg
    t = verify_tree_buffers(otrees, L, K, B + 1)
    out = dtree.verify(t, tg.cuda())
    torch.cuda.synchronize()
    for b in range(batch):
        acc, alen, nxt = oracle.verify_greedy(otrees[b], f32(tg[b]), L)
        assert out[0][b].cpu().tolist() == acc.tolist()
        assert int(out[1][b]) == alen and int(out[2][b]) == nxt
        assert alen >= 1


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_verify_t1_parity_stochastic_batch(batch):
    wl = wk.stochastic_batch(batch)
    x, spikes = wk.draft_logits(wl)
    otrees, dl = [], []
    for b in range(batch):
        l32, ids, lps = oracle_tables(x[b], 256)
        otrees.append(oracle.ddtree(lps, ids, 256).trimmed())
        dl.append(l32)
    depth = np.zeros((batch, wl.max_nodes), np.int32)
    for b, o in enumerate(otrees):
        depth[b, :o.n] = o.depth
    tgt = wk.target_logits(wl, depth, [o.n for o in otrees], spikes)
    u = wk.uniforms(wl)
    tl = np.stack([row_lse(f32(tgt[b])) for b in range(batch)])  # oracle normalisers of every row
    t = verify_tree_buffers(otrees, 16, 256, wl.max_nodes, lse_rows=dl)
    tgt_d, x_d, u_d = tgt.cuda(), x.cuda(), u.cuda()
    out = dtree.verify(t, tgt_d, temperature=1.0, draft=x_d, uniforms=u_d,
                       target_lse=torch.from_numpy(tl).cuda())
    # and with the GPU computing the visited normalisers itself
    vlse = torch.zeros((batch, 17), device="cuda")
    out2 = dtree.verify(t, tgt_d, temperature=1.0, draft=x_d, uniforms=u_d, visited_lse=vlse)
    torch.cuda.synchronize()
    for b in range(batch):
        acc, alen, nxt, used = oracle.verify_t1(otrees[b], f32(tgt[b]), f32(x[b]), dl[b], u[b].numpy(), 16,
                                                wl.max_nodes, lse_in=tl[b])
        assert out[0][b].cpu().tolist() == acc.tolist(), b
        assert int(out[1][b]) == alen and int(out[2][b]) == nxt, b
        assert out2[0][b].cpu().tolist() == acc.tolist(), b
        assert int(out2[1][b]) == alen and int(out2[2][b]) == nxt, b
        assert np.max(np.abs(vlse[b, :alen + 1].cpu().numpy() - used[:alen + 1])) < TOL


def test_verify_t1_deep_walks_and_residual_paths():
    # target = drafter (p = q): every first child is accepted and the leaf
    # draws its bonus from P; target = -drafter: the root's children are all
    # rejected and the replacement comes from the residual.
    batch, L, V, K, B = 2, 6, 2000, 4, 30
    x = gen_logits(batch, L, V, "f32", 1.0, 0.9, seed=9)
    otrees, dl = [], []
    for b in range(batch):
        l32, ids, lps = oracle_tables(x[b], K)
        otrees.append(oracle.ddtree(lps, ids, B).trimmed())
        dl.append(l32)
    t = verify_tree_buffers(otrees, L, K, B + 1, lse_rows=dl)
    for mode in ("accept", "reject"):
        tg = torch.zeros((batch, B + 1, V))
        for b, o in enumerate(otrees):
            for n in range(o.n):
                d = min(int(o.depth[n]), L - 1)
                tg[b, n] = x[b, d] if mode == "accept" else -x[b, d]
        u = torch.rand((batch, 2, B + 1), generator=torch.Generator().manual_seed(3))
        tl = np.stack([row_lse(tg[b].numpy()) for b in range(batch)])
        out = dtree.verify(t, tg.cuda(), temperature=1.0, draft=x.cuda(), uniforms=u.cuda(),
                           target_lse=torch.from_numpy(tl).cuda())
        torch.cuda.synchronize()
        for b in range(batch):
            acc, alen, nxt, _ = oracle.verify_t1(otrees[b], tg[b].numpy(), x[b].numpy(), dl[b], u[b].numpy(), L,
                                                 B + 1, lse_in=tl[b])
            assert out[0][b].cpu().tolist() == acc.tolist(), (mode, b)
            assert int(out[1][b]) == alen and int(out[2][b]) == nxt, (mode, b)


# ---------------------------------------------------------------------------
# DARTree (oracle tables fed to the GPU selection)
# ---------------------------------------------------------------------------
def dartree_case(batch, L, V, K, W, B, beta, R, root, seed, dtype="bf16", scale=3.0, x=None, U=None, Vt=None,
                 sample=None):
    if x is None:
        x = gen_logits(batch, L, V, dtype, scale, 0.7, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    if R and U is None:
        U = torch.randn((V, R), generator=g) * 0.1
        Vt = torch.randn((V, R), generator=g) * 0.1
    rt = torch.randint(0, V, (batch,), generator=g, dtype=torch.int32) if root else None
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype=dtype, K=K, W=W, B=B, beta=beta, R=R,
                     U=U.cuda() if R else None, Vt=Vt.cuda() if R else None,
                     root_tok=rt.cuda() if root else None)
    max_nodes = min(B, W * L) + 1
    tree = dtree.TreeBuffers.for_params(p, max_nodes=max_nodes)
    sample = list(range(batch)) if sample is None else sample
    tables = {}
    dtree.candidates(p, x.cuda(), tree)  # non-sampled requests keep the GPU's own tables
    for b in sample:
        tables[b] = oracle_tables(x[b], K)
        upload_tables(tree, b, *tables[b])
    dtree.select(p, tree, workspace=dtree.make_workspace(p))
    torch.cuda.synchronize()
    for b in sample:
        _, ids, lps = tables[b]
        ot, info, _ = oracle.dartree(lps, ids, U.numpy() if R else None, Vt.numpy() if R else None,
                                     int(rt[b]) if root else -1, W, beta, B, Mmax=max_nodes)
        assert_same_tree(gpu_tree(tree, b), ot.trimmed(), "dartree b=%d" % b)
        st = int(tree.status[b])
        assert (st >> dtree.DT_DEV_VIOLATION_SHIFT) == min(info["violations"], (1 << 23) - 1)
        assert bool(st & dtree.DT_DEV_BESTFIRST) == (not info["topb_equals_bestfirst"])
    return tree, p


@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_dartree_parity_small(beta):
    dartree_case(3, 6, 2000, 8, 6, 20, beta, 16, True, seed=1)
    dartree_case(2, 5, 900, 5, 7, 35, beta, 0, False, seed=2)       # no correction term
    dartree_case(2, 4, 300, 3, 9, 200, beta, 8, False, seed=3)      # B above |S|
    dartree_case(2, 6, 700, 16, 32, 100, beta, 64, True, seed=4)    # W*K = 512 candidates per depth


def test_dartree_parity_non_monotone_fallback():
    # a constant positive Markov term (<U, Vt> = 8 for every pair) makes every
    # child outscore its parent, so TopB(S) lists children before parents: the
    # result is the best-first heap over S, and the status word says so
    batch, L, V, K, W, B = 2, 6, 400, 4, 5, 12
    x = gen_logits(batch, L, V, "f32", 2.0, 0.5, seed=4)
    U = torch.ones((V, 8))
    Vt = torch.ones((V, 8))
    tree, _ = dartree_case(batch, L, V, K, W, B, 0.0, 8, False, seed=8, dtype="f32", x=x, U=U, Vt=Vt)
    for b in range(batch):
        st = int(tree.status[b])
        assert st & dtree.DT_DEV_BESTFIRST
        assert (st >> dtree.DT_DEV_VIOLATION_SHIFT) > 0


@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_dartree_full_size(beta):
    wl = wk.dartree_supertree(beta)
    x, spikes = wk.draft_logits(wl)
    U, Vt = wk.markov_tables(wl.V, wl.R)
    tree, p = dartree_case(wl.batch, wl.L, wl.V, wl.K, wl.W, wl.B, beta, wl.R, False, seed=0, x=x, U=U, Vt=Vt,
                           sample=[0, 3, 7])
    for b in range(wl.batch):
        assert int(tree.n_nodes[b]) - 1 == 16 + 15 * 32  # |S| = 496 < B: T = S
    # end to end for every request (GPU tables) against the oracle from raw logits
    t2 = dtree.TreeBuffers.for_params(p, max_nodes=tree.max_nodes)
    dtree.build_tree(p, x.cuda(), t2, workspace=dtree.make_workspace(p))
    torch.cuda.synchronize()
    for b in (0, 5):
        _, ids, lps = oracle_tables(x[b], wl.K)
        ot, _, _ = oracle.dartree(lps, ids, U.numpy(), Vt.numpy(), -1, wl.W, beta, wl.B, Mmax=tree.max_nodes)
        E = oracle.markov_table(ids, U.numpy(), Vt.numpy(), -1)
        check_end_to_end(gpu_tree(t2, b), ot.trimmed(), lps, "dartree", E=E, beta=beta,
                         what="dartree beta=%g b=%d" % (beta, b))


# ---------------------------------------------------------------------------
# TALON (oracle tables fed to the GPU selection)
# ---------------------------------------------------------------------------
def talon_case(x, N, mu, talon_k=10, sample=None):
    batch, L, V = x.shape
    p = dtree.Params(mode="talon", batch=batch, L=L, V=V, dtype="bf16" if x.dtype == torch.bfloat16 else "f32",
                     talon_k=min(talon_k, N), mu=mu, N=N)
    tree = dtree.TreeBuffers.for_params(p)
    dtree.candidates(p, x.cuda(), tree)
    sample = list(range(batch)) if sample is None else sample
    want, tables = {}, {}
    log_mu = p.struct().log_mu
    for b in sample:
        l32, ids, lps = oracle_tables(x[b], p.Kc)
        upload_tables(tree, b, l32, ids, lps)
        want[b] = oracle.talon(lps, ids, p.talon_k, log_mu, N).trimmed()
        tables[b] = lps
    dtree.select(p, tree)
    torch.cuda.synchronize()
    for b in sample:
        assert_same_tree(gpu_tree(tree, b), want[b], "talon b=%d" % b)
    return tree, p, want, tables


@pytest.mark.parametrize("N,mu,scale", [(7, 0.25, 3.0), (60, 0.03, 3.0), (200, 0.01, 0.5), (1024, 0.03, 0.7),
                                        (1024, 1e-4, 0.2), (1, 0.5, 3.0), (1024, 0.5, 0.01)])
def test_talon_parity_small(N, mu, scale):
    x = gen_logits(3, 8, 3000, "bf16", scale, 0.6, seed=N)
    talon_case(x, N, mu)


@pytest.mark.parametrize("N", [30, 257])
def test_talon_layer_overflow_all_ties(N):
    # equal logits: every child of a layer scores the same, so the budget cut
    # falls inside one run of ties, broken by the lexicographic order
    x = torch.full((2, 6, 500), 0.5).to(torch.bfloat16)
    x[1, :, 7] = 1.0  # second request: one favoured token per position
    talon_case(x, N, 0.5, talon_k=4)


@pytest.mark.parametrize("N", [60, 1024])
def test_talon_full_size(N):
    wl = wk.talon_gated(N)
    x, spikes = wk.draft_logits(wl)
    sample = [0, 17, 40, 63]
    tree, p, want, tables = talon_case(x, N, 0.03, sample=sample)
    # mask of the sampled oracle trees through the GPU, and greedy verify
    t2 = dtree.TreeBuffers(len(sample), wl.L, wl.Kc, wl.max_nodes)
    for i, b in enumerate(sample):
        upload_tree(t2, i, want[b])
    mask, pos = dtree.alloc_mask(t2)
    dtree.tree_mask(t2, mask, pos)
    depth = np.zeros((len(sample), wl.max_nodes), np.int32)
    for i, b in enumerate(sample):
        depth[i, :want[b].n] = want[b].depth
    tgt = wk.target_logits(wl, depth, [want[b].n for b in sample], spikes[sample])
    out = dtree.verify(t2, tgt.cuda())
    torch.cuda.synchronize()
    for i, b in enumerate(sample):
        o = want[b]
        rc, om, _ = oracle.tree_mask(o, wl.max_nodes, wl.L)
        assert rc == 0 and np.array_equal(mask[i].cpu().numpy().view(np.uint32)[:o.n], om[:o.n])
        acc, alen, nxt = oracle.verify_greedy(o, f32(tgt[i]), wl.L)
        assert out[0][i].cpu().tolist() == acc.tolist()
        assert int(out[1][i]) == alen and int(out[2][i]) == nxt
    # end to end from raw logits (GPU alone) on the same sample
    t3 = dtree.TreeBuffers.for_params(p)
    dtree.build_tree(p, x.cuda(), t3)
    torch.cuda.synchronize()
    log_mu = p.struct().log_mu
    for b in sample:
        check_end_to_end(gpu_tree(t3, b), want[b], tables[b], "talon", log_mu=log_mu, what="talon N=%d b=%d" % (N, b))


# ---------------------------------------------------------------------------
# Mask written by the selection kernel itself (dt_build_tree_mask)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["ddtree", "dartree", "talon", "talon_large"])
def test_fused_mask_equals_mask_kernel(mode):
    batch, L, V = 3, 8, 5000
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=77).cuda()
    if mode == "ddtree":
        p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype="bf16", K=40, B=40)
    elif mode == "dartree":
        g = torch.Generator().manual_seed(78)
        U = (torch.randn((V, 64), generator=g) * 0.1).cuda()
        Vt = (torch.randn((V, 64), generator=g) * 0.1).cuda()
        p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype="bf16", K=8, W=16, B=60, beta=-0.25, R=64,
                         U=U, Vt=Vt)
    elif mode == "talon":
        p = dtree.Params(mode="talon", batch=batch, L=L, V=V, dtype="bf16", talon_k=6, mu=0.05, N=90)
    else:  # more than 512 rows: mask rows of 22 words
        p = dtree.Params(mode="talon", batch=batch, L=L, V=V, dtype="bf16", talon_k=10, mu=0.01, N=700)
    max_nodes = min(p.B, p.W * L) + 1 if mode == "dartree" else p.budget + 1
    ws = dtree.make_workspace(p)
    t1 = dtree.TreeBuffers.for_params(p, max_nodes=max_nodes)
    t2 = dtree.TreeBuffers.for_params(p, max_nodes=max_nodes)
    m1, p1 = dtree.alloc_mask(t1)
    m2, p2 = dtree.alloc_mask(t2)
    dtree.build_tree(p, x, t1, workspace=ws)
    dtree.tree_mask(t1, m1, p1, pos_offset=11)
    dtree.build_tree_mask(p, x, t2, m2, p2, workspace=ws, pos_offset=11)
    torch.cuda.synchronize()
    for f in ("node_tok", "parent", "depth", "rank", "n_nodes", "status"):
        assert torch.equal(getattr(t1, f), getattr(t2, f)), (mode, f)
    for b in range(batch):
        n = int(t1.n_nodes[b])
        assert torch.equal(m1[b, :n], m2[b, :n]), (mode, b)
        assert torch.equal(p1[b, :n], p2[b, :n]), (mode, b)


def test_fused_mask_single_request_against_oracle():
    wl = wk.single_request(256)
    x, _ = wk.draft_logits(wl)
    p = dtree.Params(mode="ddtree", batch=1, L=16, V=wl.V, dtype="bf16", K=256, B=256)
    # the oracle side: its own stage 1, tree and mask
    _, _, ids, lps = oracle.candidates(f32(x[0]), 256)
    ot = oracle.ddtree(lps, ids, 256, Mmax=257)
    rc, omask, opos = oracle.tree_mask(ot, 257, 16, pos_offset=5)
    assert rc == 0
    # the GPU side: stage 1, selection and the fused mask from the same logits
    t = dtree.TreeBuffers.for_params(p)
    m, pp = dtree.alloc_mask(t)
    dtree.build_tree_mask(p, x.cuda(), t, m, pp, pos_offset=5)
    torch.cuda.synchronize()
    g = gpu_tree(t, 0)
    n = g.n
    # the mask of the GPU's own tree, always (the oracle's mask builder on the GPU's parents and depths)
    rc, gmask, gpos = oracle.tree_mask(g, 257, 16, pos_offset=5)
    assert rc == 0
    assert np.array_equal(m[0, :n].cpu().numpy().view(np.uint32), gmask[:n])
    assert np.array_equal(pp[0, :n].cpu().numpy(), gpos[:n])
    # and the tree against the oracle's: near-ties only; where the two agree node for node, the masks too
    check_end_to_end(g, ot.trimmed(), lps, "ddtree", what="fused mask single request")
    if g.n == ot.n and np.array_equal(g.tok, ot.tok[:n]) and np.array_equal(g.parent, ot.parent[:n]):
        assert np.array_equal(m[0, :n].cpu().numpy().view(np.uint32), omask[:n])
        assert np.array_equal(pp[0, :n].cpu().numpy(), opos[:n])
