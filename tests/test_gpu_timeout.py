"""The timeout path of the bounded waits, on the GPU, without a fault.

Every mbarrier wait in the library has a bound; when it runs out the kernel
records it and finishes (stage 1 writes a NaN normaliser, which the selection
turns into DT_DEV_TIMEOUT; the walk sets DT_DEV_TIMEOUT; the normaliser writes
NaN).  dt_test_wait_fault makes a kernel first wait, with a short bound, on a
barrier that nothing completes -- the wait runs out every time -- and then on
its real copy as usual, so every copy lands before its data is read.  Each
test checks the flag, then turns the hook off and checks that the same call
on the same context gives the oracle's result again."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from test_gpu_parity import assert_same_tree, f32, gen_logits, gpu_tree, oracle_tables, upload_tables, upload_tree

pytestmark = pytest.mark.gpu

BUDGET = 2_000_000  # SM clock cycles, about a millisecond


@pytest.fixture(autouse=True)
def _hook_off(cuda_lib):
    dtree.set_test_wait_fault(())
    yield
    dtree.set_test_wait_fault(())


def test_hook_rejects_bad_arguments(cuda_lib):
    assert cuda_lib.dt_test_wait_fault(0x8, BUDGET) == -1
    assert cuda_lib.dt_test_wait_fault(0x1, 0) == -1
    assert cuda_lib.dt_test_wait_fault(0x1, (1 << 28) + 1) == -1
    assert cuda_lib.dt_test_wait_fault(0, 0) == 0


def test_stage1_timeout_sets_nan_normaliser_and_status():
    batch, L, V, K = 2, 4, 5000, 16
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=3).cuda()
    p = dtree.Params(mode="ddtree", batch=batch, L=L, V=V, dtype="bf16", K=K, B=K)
    assert dtree.stage1_plan(p)[0] == "cluster"
    tree = dtree.TreeBuffers.for_params(p)
    dtree.set_test_wait_fault(("stage1",), BUDGET)
    dtree.build_tree(p, x, tree)
    torch.cuda.synchronize()
    assert torch.isnan(tree.lse).all()
    assert all(int(s) & dtree.DT_DEV_TIMEOUT for s in tree.status.cpu())
    # hook off: the same call on the same context is clean and equals the oracle
    dtree.set_test_wait_fault(())
    tree2 = dtree.TreeBuffers.for_params(p)
    dtree.build_tree(p, x, tree2)
    torch.cuda.synchronize()
    assert int(tree2.status.abs().sum()) == 0 and torch.isfinite(tree2.lse).all()
    for b in range(batch):
        _, ids, lps = oracle_tables(x[b].cpu(), K)
        assert np.array_equal(tree2.cand_id[b].cpu().numpy(), ids)


def test_walk_timeout_sets_status():
    L, V, K, B = 4, 3000, 6, 20
    x = gen_logits(1, L, V, "bf16", 3.0, 0.7, seed=4)
    _, ids, lps = oracle_tables(x[0], K)
    o = oracle.ddtree(lps, ids, B).trimmed()
    tree = dtree.TreeBuffers(1, L, K, B + 1)
    upload_tree(tree, 0, o)
    tgt = gen_logits(1, B + 1, V, "bf16", 3.0, 0.7, seed=5)
    dtree.set_test_wait_fault(("walk",), BUDGET)
    dtree.verify(tree, tgt.cuda())
    torch.cuda.synchronize()
    assert int(tree.status[0]) & dtree.DT_DEV_TIMEOUT
    dtree.set_test_wait_fault(())
    tree.status.zero_()
    out = dtree.verify(tree, tgt.cuda())
    torch.cuda.synchronize()
    assert int(tree.status[0]) == 0
    acc, alen, nxt = oracle.verify_greedy(o, f32(tgt[0]), L)
    assert out[0][0].cpu().tolist() == acc.tolist() and int(out[1][0]) == alen and int(out[2][0]) == nxt


def test_normaliser_timeout_reaches_the_selection():
    batch, L, V, K = 1, 3, 2000, 8
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=6)
    g = torch.Generator().manual_seed(7)
    U = (torch.randn((V, 64), generator=g) * 0.1).cuda()
    Vt = (torch.randn((V, 64), generator=g) * 0.1).cuda()
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype="bf16", K=K, W=8, B=20, beta=-0.25, R=64,
                     U=U, Vt=Vt, markov_norm=True)
    tree = dtree.TreeBuffers.for_params(p, max_nodes=21)
    ws = dtree.make_workspace(p)
    dtree.set_test_wait_fault(("normaliser",), BUDGET)
    dtree.build_tree(p, x.cuda(), tree, workspace=ws)
    torch.cuda.synchronize()
    z = dtree.znorm_view(p, ws)
    assert torch.isnan(z[0, 1:]).all()  # rows with a parent token
    assert int(tree.status[0]) & dtree.DT_DEV_TIMEOUT
    dtree.set_test_wait_fault(())
    dtree.build_tree(p, x.cuda(), tree, workspace=ws)
    torch.cuda.synchronize()
    assert int(tree.status[0]) == 0 and torch.isfinite(dtree.znorm_view(p, ws)).all()
