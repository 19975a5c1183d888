"""GPU edge cases of the later rows against the oracle: a root-only tree under
every walk rule, a one-candidate chain and a one-node budget in the heap,
per-request budgets outside [1, B] (clamped), SABA with a one-value range and
one position, and DARTree (fixed) with the normalised correction; and the tie
and boundary rules the oracle's pins fix: a greedy tie across the vocabulary
goes to the smaller id, a uniform of exactly 1/2 over two equal masses draws
the second token, SABA takes the smallest of tied budgets, and a child that
scores exactly its parent's score (a certain position) follows its parent."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from test_gpu_parity import assert_same_tree, dartree_case, f32, gen_logits, gpu_tree, oracle_tables, talon_case, \
    upload_tables, verify_tree_buffers

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _root_only():
    return oracle.Tree(np.array([-1], np.int32), np.array([-1], np.int32), np.array([0], np.int32),
                       np.array([-1], np.int32), np.zeros(1, np.float32), 1)


@pytest.mark.parametrize("rule", ["greedy", "ratio", "iter_residual", "target_match", "markov"])
def test_root_only_tree_every_rule(rule):
    # nothing to accept: the walk emits one token from the root's target row
    batch, L, V, Mmax = 2, 4, 3001, 5
    x = gen_logits(batch, L, V, "f32", 2.0, 0.5, seed=3)
    dl = [oracle_tables(x[b], 4)[0] for b in range(batch)]
    t = verify_tree_buffers([_root_only()] * batch, L, 4, Mmax, lse_rows=dl)
    tg = torch.randn((batch, Mmax, V), generator=torch.Generator().manual_seed(4)) * 2
    u = torch.rand((batch, 2, Mmax), generator=torch.Generator().manual_seed(5))
    U = torch.randn((V, 64), generator=torch.Generator().manual_seed(6)) * 0.1
    z = np.zeros((batch, L, 4), np.float32)
    if rule == "greedy":
        out = dtree.verify(t, tg.cuda())
    elif rule == "markov":
        p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype="f32", K=4, W=4, B=4, R=64, U=U.cuda(),
                         Vt=U.cuda(), root_tok=torch.tensor([7, 9], dtype=torch.int32).cuda(), markov_norm=True)
        out = dtree.verify_markov(p, t, tg.cuda(), x.cuda(), torch.from_numpy(z).cuda(), u.cuda())
    else:
        out = dtree.verify(t, tg.cuda(), draft=x.cuda(), uniforms=u.cuda(), rule=rule)
    torch.cuda.synchronize()
    for b in range(batch):
        if rule == "greedy":
            want = oracle.verify_greedy(_root_only(), tg[b].numpy(), L)
        elif rule == "markov":
            want = oracle.verify_t1_markov(_root_only(), tg[b].numpy(), f32(x[b]), dl[b], U.numpy(), U.numpy(),
                                           [7, 9][b], z[b], u[b].numpy(), L, Mmax)
        else:
            want = oracle.verify_t1(_root_only(), tg[b].numpy(), f32(x[b]), dl[b], u[b].numpy(), L, Mmax,
                                    rule=rule)
        assert out[0][b].cpu().tolist() == want[0].tolist() and int(out[1][b]) == 0 and int(out[2][b]) == want[2]


@pytest.mark.parametrize("K,B", [(1, 6), (5, 1)])
def test_heap_chain_and_single_node(K, B):
    batch, L, V = 2, 6, 900
    x = gen_logits(batch, L, V, "bf16", 2.0, 0.7, seed=K + B)
    g = torch.Generator().manual_seed(8)
    U = torch.randn((V, 64), generator=g) * 0.2
    Vt = torch.randn((V, 64), generator=g) * 0.2
    p = dtree.Params(mode="heap", batch=batch, L=L, V=V, dtype="bf16", K=K, B=B, R=64, U=U.cuda(), Vt=Vt.cuda())
    tree = dtree.TreeBuffers.for_params(p)
    ws = dtree.make_workspace(p)
    tabs = {b: oracle_tables(x[b], K) for b in range(batch)}
    for b in range(batch):
        upload_tables(tree, b, *tabs[b])
    dtree.select(p, tree, workspace=ws)
    torch.cuda.synchronize()
    for b in range(batch):
        _, ids, lps = tabs[b]
        want = oracle.heap_select(lps, ids, B, E=oracle.markov_table(ids, U.numpy(), Vt.numpy(), -1))
        got = gpu_tree(tree, b)
        assert_same_tree(got, want, "heap K=%d B=%d" % (K, B))
        assert got.n == min(B, L if K == 1 else B) + 1


def test_per_request_budgets_are_clamped():
    batch, L, V, K, B = 4, 8, 2000, 16, 40
    x = gen_logits(batch, L, V, "bf16", 2.0, 0.7, seed=12)
    budgets = torch.tensor([0, -5, 1000, 7], dtype=torch.int32)
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=B, budgets=budgets.cuda())
    tree = dtree.TreeBuffers.for_params(p)
    tabs = {b: oracle_tables(x[b], K) for b in range(batch)}
    for b in range(batch):
        upload_tables(tree, b, *tabs[b])
    dtree.select(p, tree)
    torch.cuda.synchronize()
    for b, want_b in enumerate([1, 1, B, 7]):
        assert_same_tree(gpu_tree(tree, b), oracle.ddtree(tabs[b][2], tabs[b][1], want_b), "budget %d" % want_b)


def test_saba_fixed_range_and_one_position():
    batch, L, V, K = 3, 1, 500, 8
    x = gen_logits(batch, L, V, "bf16", 2.0, 0.7, seed=13)
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=16)
    tree = dtree.TreeBuffers.for_params(p)
    tabs = {b: oracle_tables(x[b], K) for b in range(batch)}
    for b in range(batch):
        upload_tables(tree, b, *tabs[b])
    st = dtree.SabaState(batch, 3)
    budget = torch.zeros(batch, dtype=torch.int32, device="cuda")
    state = torch.zeros((batch, 4), device="cuda")
    hidden = torch.randn((batch, L, 32), generator=torch.Generator().manual_seed(2)).cuda()
    dtree.saba_budget(tree, st, 0.5, 10.0, 9, 9, budget, state, hidden=hidden,
                      prev_acc_len=torch.tensor([2, 0, 5], dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    assert budget.cpu().tolist() == [9, 9, 9]
    s = state.cpu().numpy()
    assert np.all(s[:, 1] == 0.0)  # one position: no adjacent pair
    assert s[:, 2].tolist() == [2.0, 0.0, 5.0] and s[:, 3].tolist() == [3.0, 1.0, 6.0]


def test_dartree_fixed_with_normalised_correction():
    batch, L, V, K, B = 2, 8, 3000, 16, 20
    x = gen_logits(batch, L, V, "bf16", 2.0, 0.7, seed=21)
    g = torch.Generator().manual_seed(22)
    U = torch.randn((V, 64), generator=g) * 0.1
    Vt = torch.randn((V, 64), generator=g) * 0.1
    rt = torch.randint(0, V, (batch,), generator=g, dtype=torch.int32)
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=B, R=64, U=U.cuda(), Vt=Vt.cuda(),
                     root_tok=rt.cuda(), markov_norm=True, budget_policy="uniform")
    tree = dtree.TreeBuffers.for_params(p, max_nodes=B + 1)
    ws = dtree.make_workspace(p)
    zv = dtree.znorm_view(p, ws)
    w = oracle.uniform_widths(B, L)
    want = {}
    for b in range(batch):
        tab = oracle_tables(x[b], K)
        upload_tables(tree, b, *tab)
        z = oracle.markov_norm(f32(x[b]), tab[1], U.numpy(), Vt.numpy(), int(rt[b]))
        zv[b].copy_(torch.from_numpy(z))
        t, info, _ = oracle.dartree(tab[2], tab[1], U.numpy(), Vt.numpy(), int(rt[b]), int(w.max()), 0.0, B,
                                    Mmax=B + 1, znorm=z, widths=w)
        assert info["violations"] == 0  # normalised: no edge raises the score
        want[b] = t.trimmed()
    dtree.select(p, tree, workspace=ws)
    torch.cuda.synchronize()
    for b in range(batch):
        assert_same_tree(gpu_tree(tree, b), want[b], "fixed normalised b=%d" % b)


def test_greedy_tie_goes_to_the_smaller_id():
    # the two equal maxima sit far apart in the row (different CTAs of the walk's
    # cluster); the root's children carry the larger id first in rank order
    batch, L, V, Mmax = 2, 3, 3001, 3
    t = oracle.Tree(np.array([-1, 2900, 17], np.int32), np.array([-1, 0, 0], np.int32),
                    np.array([0, 1, 1], np.int32), np.array([-1, 0, 1], np.int32), np.zeros(3, np.float32), 3)
    tg = torch.randn((batch, Mmax, V), generator=torch.Generator().manual_seed(7))
    tg[:, 0, [17, 2900]] = 9.0
    tg[:, 2, 123] = 9.0
    tg[:, 1, 456] = 9.0
    tb = verify_tree_buffers([t] * batch, L, 2, Mmax)
    out = dtree.verify(tb, tg.cuda())
    torch.cuda.synchronize()
    for b in range(batch):
        want = oracle.verify_greedy(t, tg[b].numpy(), L)
        assert want[1] == 1 and want[0][1] == 2 and want[2] == 123
        assert out[0][b].cpu().tolist()[:2] == [0, 2] and int(out[1][b]) == 1 and int(out[2][b]) == 123


@pytest.mark.parametrize("rule", ["ratio", "target_match"])
def test_draw_at_a_mass_boundary_takes_the_next_token(rule):
    batch, L, V, Mmax = 4, 4, 3001, 1
    x = gen_logits(batch, L, V, "f32", 2.0, 0.5, seed=31)
    dl = [oracle_tables(x[b], 4)[0] for b in range(batch)]
    tg = torch.full((batch, Mmax, V), -30.0)
    tg[:, 0, [5, 2000]] = 1.5  # two equal masses; every other token's mass rounds to 0
    u = torch.zeros((batch, 2, Mmax))
    u[:, 1, 0] = torch.tensor([0.5, 0.4999999, 0.0, 0.9999999])
    root = oracle.Tree(np.array([-1], np.int32), np.array([-1], np.int32), np.array([0], np.int32),
                       np.array([-1], np.int32), np.zeros(1, np.float32), 1)
    tb = verify_tree_buffers([root] * batch, L, 4, Mmax, lse_rows=dl)
    out = dtree.verify(tb, tg.cuda(), draft=x.cuda(), uniforms=u.cuda(), rule=rule)
    torch.cuda.synchronize()
    for b, tok in enumerate([2000, 5, 5, 2000]):
        want = oracle.verify_t1(root, tg[b].numpy(), f32(x[b]), dl[b], u[b].numpy(), L, Mmax, rule=rule)
        assert want[2] == tok, (b, want[2])
        assert int(out[1][b]) == 0 and int(out[2][b]) == tok, (rule, b, int(out[2][b]))


def test_saba_tie_takes_the_smaller_budget():
    # c_fixed / c_verify = 1000.5: budgets 1000 and 1001 score the same in fp32
    batch, L, V, K = 2, 4, 500, 8
    x = gen_logits(batch, L, V, "bf16", 2.0, 0.7, seed=17)
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=16)
    tree = dtree.TreeBuffers.for_params(p)
    tabs = {b: oracle_tables(x[b], K) for b in range(batch)}
    for b in range(batch):
        upload_tables(tree, b, *tabs[b])
    st = dtree.SabaState(batch, 4)
    budget = torch.zeros(batch, dtype=torch.int32, device="cuda")
    state = torch.zeros((batch, 4), device="cuda")
    dtree.saba_budget(tree, st, 1.0, 1000.5, 1, 1024, budget, state)
    torch.cuda.synchronize()
    for b in range(batch):
        want, _ = oracle.saba(tabs[b][2][:, 0], None, oracle.SabaState(4), -1, 1.0, 1000.5, 1, 1024)
        assert want == 1000 and int(budget[b]) == 1000


def _certain_second_position(batch, L, V, seed):
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.0, seed=seed)
    x[:, 1, :] = -30.0
    x[:, 1, 11] = 0.0  # lp = -2.8e-10: a depth-2 child of token 11 keeps its parent's fp32 score
    return x


def _has_equal_score_edges(t):
    return sum(int(t.score[n] == t.score[t.parent[n]]) for n in range(1, t.n) if t.parent[n] > 0)


def test_equal_parent_and_child_scores_keep_the_parent_first():
    x = _certain_second_position(2, 6, 3000, seed=41)
    tree, p, want, _ = talon_case(x, 40, 0.2, talon_k=4)
    for b in range(2):
        g = gpu_tree(tree, b)
        assert _has_equal_score_edges(g) >= 1
        assert all(g.parent[n] < n for n in range(1, g.n))
    tree, _ = dartree_case(2, 6, 3000, 8, 6, 20, 0.0, 0, False, seed=42, x=x)
    for b in range(2):
        g = gpu_tree(tree, b)
        assert _has_equal_score_edges(g) >= 2
        assert all(g.parent[n] < n for n in range(1, g.n))
