"""GPU parity of the budget policies against the oracle: DARTree (fixed)'s
uniform per-depth widths, per-request budgets in the DDTree and heap
selections, and SABA's state and budgets over several rounds.  Inputs flow
from the oracle to the GPU."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from test_gpu_parity import assert_same_tree, f32, gen_logits, gpu_tree, oracle_tables, upload_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


@pytest.mark.parametrize("B,K", [(64, 64), (70, 16), (512, 16)])
def test_dartree_fixed_uniform_widths(B, K):
    batch, L, V = 3, 16, 20000
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=B + K)
    g = torch.Generator().manual_seed(B)
    U = torch.randn((V, 64), generator=g) * 0.1
    Vt = torch.randn((V, 64), generator=g) * 0.1
    rt = torch.randint(0, V, (batch,), generator=g, dtype=torch.int32)
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=B, R=64, U=U.cuda(), Vt=Vt.cuda(),
                     root_tok=rt.cuda(), budget_policy="uniform")
    tree = dtree.TreeBuffers.for_params(p, max_nodes=B + 1)
    ws = dtree.make_workspace(p)
    tabs = {}
    for b in range(batch):
        tabs[b] = oracle_tables(x[b], K)
        upload_tables(tree, b, *tabs[b])
    dtree.select(p, tree, workspace=ws)
    torch.cuda.synchronize()
    w = oracle.uniform_widths(B, L)
    for b in range(batch):
        o, info, _ = oracle.dartree(tabs[b][2], tabs[b][1], U.numpy(), Vt.numpy(), int(rt[b]), int(w.max()), 0.0, B,
                                    Mmax=B + 1, widths=w)
        assert_same_tree(gpu_tree(tree, b), o.trimmed(), "dartree fixed b=%d" % b)
        assert info["supertree_size"] == o.n - 1  # the uniform widths sum to B: nothing is pruned


def test_per_request_budgets_ddtree_and_heap():
    batch, L, V, K, B = 6, 16, 30000, 64, 64
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=5)
    budgets = torch.tensor([64, 1, 17, 40, 63, 2], dtype=torch.int32)
    g = torch.Generator().manual_seed(6)
    U = torch.randn((V, 64), generator=g) * 0.1
    Vt = torch.randn((V, 64), generator=g) * 0.1
    tabs = {b: oracle_tables(x[b], K) for b in range(batch)}
    for mode in ("ddtree", "heap"):
        kw = dict(R=64, U=U.cuda(), Vt=Vt.cuda()) if mode == "heap" else {}
        p = dtree.Params(mode=mode, batch=batch, L=L, V=V, dtype="bf16", K=K, B=B, budgets=budgets.cuda(), **kw)
        tree = dtree.TreeBuffers.for_params(p, max_nodes=B + 1)
        ws = dtree.make_workspace(p)
        for b in range(batch):
            upload_tables(tree, b, *tabs[b])
        dtree.select(p, tree, workspace=ws)
        torch.cuda.synchronize()
        for b in range(batch):
            _, ids, lps = tabs[b]
            Bb = int(budgets[b])
            if mode == "ddtree":
                o = oracle.ddtree(lps, ids, Bb)
            else:
                o = oracle.heap_select(lps, ids, Bb, E=oracle.markov_table(ids, U.numpy(), Vt.numpy(), -1))
            gt = gpu_tree(tree, b)
            assert gt.n == Bb + 1, (mode, b)
            assert_same_tree(gt, o, "%s budget %d" % (mode, Bb))
            assert np.array_equal(gt.score[:gt.n], o.score[:o.n])


def test_saba_rounds_match_the_oracle():
    batch, L, V, K, Hd, w = 5, 16, 8000, 32, 512, 4
    rng = np.random.default_rng(0)
    st_g = dtree.SabaState(batch, w)
    st_o = [oracle.SabaState(w) for _ in range(batch)]
    budget = torch.zeros(batch, dtype=torch.int32, device="cuda")
    state = torch.zeros((batch, 4), device="cuda")
    cv, cf = 0.37, 29.0
    for rnd in range(7):
        x = gen_logits(batch, L, V, "bf16", 2.0, 0.6, seed=100 + rnd)
        p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=64)
        tree = dtree.TreeBuffers.for_params(p)
        tabs = {b: oracle_tables(x[b], K) for b in range(batch)}
        for b in range(batch):
            upload_tables(tree, b, *tabs[b])
        hidden = torch.randn((batch, L, Hd), generator=torch.Generator().manual_seed(rnd)).float()
        hidden[:, 1:] += hidden[:, :-1] * 0.8  # adjacent positions alike
        prev = None if rnd == 0 else torch.from_numpy(rng.integers(0, 17, batch).astype(np.int32))
        dtree.saba_budget(tree, st_g, cv, cf, 1, 256, budget, state, hidden=hidden.cuda(),
                          prev_acc_len=None if prev is None else prev.cuda())
        torch.cuda.synchronize()
        for b in range(batch):
            want_b, want_s = oracle.saba(tabs[b][2][:, 0], hidden[b].numpy(), st_o[b], -1 if prev is None else
                                         int(prev[b]), cv, cf, 1, 256)
            got = state[b].cpu().numpy()
            assert int(budget[b]) == want_b, (rnd, b)
            assert got[2] == want_s[2] and got[3] == want_s[3], (rnd, b)  # hist, a: exact
            assert abs(got[0] - want_s[0]) < 1e-5 and abs(got[1] - want_s[1]) < 1e-4, (rnd, b, got, want_s)
            assert int(st_g.count[b]) == int(st_o[b].count[0])
            assert st_g.ring[b].cpu().tolist() == st_o[b].ring.tolist()
    # the printed model's optimum c_fixed / c_verify = 78.4, whatever the state
    assert set(budget.cpu().tolist()) <= {78, 79}


def test_saba_budgets_drive_the_build():
    batch, L, V, K = 4, 16, 151936, 128
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=9).cuda()
    budget = torch.zeros(batch, dtype=torch.int32, device="cuda")
    state = torch.zeros((batch, 4), device="cuda")
    st = dtree.SabaState(batch, 8)
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=128, budgets=budget)
    tree = dtree.TreeBuffers.for_params(p)
    dtree.candidates(p, x, tree)
    dtree.saba_budget(tree, st, 0.5, 48.0, 8, 128, budget, state)
    dtree.select(p, tree)
    torch.cuda.synchronize()
    assert budget.cpu().tolist() == [96] * batch
    assert tree.n_nodes.cpu().tolist() == [97] * batch
