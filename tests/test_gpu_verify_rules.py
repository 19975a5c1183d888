"""GPU parity of the two further T=1 walks (dt_verify_rule) against the oracle.

DT_VERIFY_ITER_RESIDUAL (one residual per rejected sibling) and
DT_VERIFY_TARGET_MATCH (exact target-sample matching) must reproduce the
oracle's accepted path and emitted token bit for bit on the same trees,
logits, normalisers and uniforms.  Inputs flow from the oracle to the GPU."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from speculative_decoding_draft_bf16_gb300 import workloads as wk
from test_gpu_parity import TOL, f32, gen_logits, oracle_tables, row_lse, upload_tree, verify_tree_buffers

pytestmark = pytest.mark.gpu

RULES = ["iter_residual", "target_match"]


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _check(out, b, want, what):
    acc, alen, nxt = want[:3]
    assert out[0][b].cpu().tolist() == acc.tolist(), (what, b, out[0][b].cpu().tolist(), acc.tolist())
    assert int(out[1][b]) == alen and int(out[2][b]) == nxt, (what, b, int(out[1][b]), alen, int(out[2][b]), nxt)


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("batch", [1, 16])
def test_rules_full_size_stochastic_batch(rule, batch):
    # the T=1 workload shape: DDTree K=B=256 trees over V=151936, bf16
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
    tl = np.stack([row_lse(f32(tgt[b])) for b in range(batch)])
    t = verify_tree_buffers(otrees, 16, 256, wl.max_nodes, lse_rows=dl)
    tgt_d, x_d, u_d = tgt.cuda(), x.cuda(), u.cuda()
    out = dtree.verify(t, tgt_d, draft=x_d, uniforms=u_d, target_lse=torch.from_numpy(tl).cuda(), rule=rule)
    vlse = torch.zeros((batch, 17), device="cuda")
    out2 = dtree.verify(t, tgt_d, draft=x_d, uniforms=u_d, visited_lse=vlse, rule=rule)
    torch.cuda.synchronize()
    for b in range(batch):
        want = oracle.verify_t1(otrees[b], f32(tgt[b]), f32(x[b]), dl[b], u[b].numpy(), 16, wl.max_nodes,
                                lse_in=tl[b], rule=rule)
        _check(out, b, want, rule)
        _check(out2, b, want, rule + " own normalisers")
        alen, used = want[1], want[3]
        assert np.max(np.abs(vlse[b, :alen + 1].cpu().numpy() - used[:alen + 1])) < TOL


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("dtype,V", [("f32", 2000), ("bf16", 10001)])
def test_rules_deep_walks_and_residual_paths(rule, dtype, V):
    # accept: target = drafter, children accepted until a leaf; reject: target =
    # -drafter, most children rejected (many residual passes at wide nodes);
    # mixed: target rows random.  Odd V gives ragged chunk ends.
    batch, L, K, B = 3, 6, 8, 60
    x = gen_logits(batch, L, V, dtype, 1.0, 0.9, seed=V)
    otrees, dl = [], []
    for b in range(batch):
        l32, ids, lps = oracle_tables(x[b], K)
        otrees.append(oracle.ddtree(lps, ids, B).trimmed())
        dl.append(l32)
    t = verify_tree_buffers(otrees, L, K, B + 1, lse_rows=dl)
    g = torch.Generator().manual_seed(V + 1)
    for mode in ("accept", "reject", "mixed", "onehot"):
        tg = torch.zeros((batch, B + 1, V))
        for b, o in enumerate(otrees):
            for n in range(o.n):
                d = min(int(o.depth[n]), L - 1)
                xd = x[b, d].float()
                if mode == "onehot":  # a mass of exactly 2^32: the residual passes recompute (P, Q)
                    tg[b, n] = -1e4
                    tg[b, n, int(torch.randint(0, V, (1,), generator=g))] = 0.0
                else:
                    tg[b, n] = xd if mode == "accept" else (-xd if mode == "reject" else torch.randn(V, generator=g) * 2)
        tg = tg.to(x.dtype)
        u = torch.rand((batch, 2, B + 1), generator=g)
        tl = np.stack([row_lse(f32(tg[b])) for b in range(batch)])
        out = dtree.verify(t, tg.cuda(), draft=x.cuda(), uniforms=u.cuda(), target_lse=torch.from_numpy(tl).cuda(),
                           rule=rule)
        torch.cuda.synchronize()
        for b in range(batch):
            want = oracle.verify_t1(otrees[b], f32(tg[b]), f32(x[b]), dl[b], u[b].numpy(), L, B + 1, lse_in=tl[b],
                                    rule=rule)
            _check(out, b, want, (rule, mode))


def test_iter_residual_many_rejected_siblings():
    # a root with 64 children, all but a few unlikely under the target: the
    # walk sums one residual per rejected child (up to 63 passes over the row)
    batch, V, K = 4, 30000, 64
    g = torch.Generator().manual_seed(44)
    x = torch.randn((batch, 1, V), generator=g) * 2.0
    otrees, dl = [], []
    for b in range(batch):
        l32, ids, lps = oracle_tables(x[b], K)
        otrees.append(oracle.ddtree(lps, ids, K).trimmed())  # L = 1: a star of the top 64
        dl.append(l32)
        assert otrees[-1].n == K + 1
    t = verify_tree_buffers(otrees, 1, K, K + 1, lse_rows=dl)
    tg = torch.randn((batch, K + 1, V), generator=g) * 2.0
    for b, o in enumerate(otrees):
        tg[b, 0, torch.from_numpy(o.tok[1:].astype(np.int64))] -= 6.0  # children under-weighted by the target
        tg[b, 0, torch.from_numpy(o.tok[1 + 50 + b:2 + 50 + b].astype(np.int64))] += 12.0  # one likely child
    u = torch.rand((batch, 2, K + 1), generator=g)
    tl = np.stack([row_lse(tg[b].numpy()) for b in range(batch)])
    for rule in ("iter_residual", "ratio"):
        out = dtree.verify(t, tg.cuda(), draft=x.cuda(), uniforms=u.cuda(), target_lse=torch.from_numpy(tl).cuda(),
                           rule=rule)
        torch.cuda.synchronize()
        for b in range(batch):
            want = oracle.verify_t1(otrees[b], tg[b].numpy(), x[b].numpy(), dl[b], u[b].numpy(), 1, K + 1,
                                    lse_in=tl[b], rule=rule)
            _check(out, b, want, rule)


@pytest.mark.parametrize("rule", RULES)
def test_rules_widest_chunks(rule):
    # V = 16 * 32400: clusters of 16 with 32400-element chunks, runs of 65
    # elements per thread (the residual passes recompute instead of caching)
    batch, L, V, K, B = 1, 3, 16 * 32400, 6, 20
    x = gen_logits(batch, L, V, "bf16", 1.0, 0.9, seed=123)
    l32, ids, lps = oracle_tables(x[0], K)
    o = oracle.ddtree(lps, ids, B).trimmed()
    t = verify_tree_buffers([o], L, K, B + 1, lse_rows=[l32])
    g = torch.Generator().manual_seed(9)
    tg = torch.zeros((1, B + 1, V))
    for n in range(o.n):
        tg[0, n] = -x[0, min(int(o.depth[n]), L - 1)].float() + torch.randn(V, generator=g) * 0.1
    tg = tg.to(torch.bfloat16)
    for seed in range(3):
        u = torch.rand((1, 2, B + 1), generator=torch.Generator().manual_seed(seed))
        out = dtree.verify(t, tg.cuda(), draft=x.cuda(), uniforms=u.cuda(), rule=rule)
        torch.cuda.synchronize()
        want = oracle.verify_t1(o, f32(tg[0]), f32(x[0]), l32, u[0].numpy(), L, B + 1, rule=rule)
        _check(out, 0, want, (rule, seed))


def test_target_match_one_hot_rows_equal_greedy():
    batch, L, V, K, B = 4, 8, 5003, 6, 80
    x = gen_logits(batch, L, V, "bf16", 2.0, 0.8, seed=71)
    otrees = []
    for b in range(batch):
        _, ids, lps = oracle_tables(x[b], K)
        otrees.append(oracle.ddtree(lps, ids, B).trimmed())
    t = verify_tree_buffers(otrees, L, K, B + 1)
    rng = np.random.default_rng(3)
    tg = torch.full((batch, B + 1, V), -1e4)
    for b, o in enumerate(otrees):
        for n in range(o.n):
            kids = [int(o.tok[c]) for c in range(1, o.n) if o.parent[c] == n]
            tok = kids[rng.integers(len(kids))] if kids and rng.random() < 0.85 else int(rng.integers(V))
            tg[b, n, tok] = 0.0
    tg = tg.to(torch.bfloat16)
    u = torch.rand((batch, 2, B + 1), generator=torch.Generator().manual_seed(5))
    out = dtree.verify(t, tg.cuda(), uniforms=u.cuda(), rule="target_match")
    torch.cuda.synchronize()
    for b in range(batch):
        acc, alen, nxt = oracle.verify_greedy(otrees[b], f32(tg[b]), L)
        _check(out, b, (acc, alen, nxt), "target_match one-hot")


def test_verify_rule_argument_checks():
    o = oracle.Tree(np.array([-1, 3], np.int32), np.array([-1, 0], np.int32), np.array([0, 1], np.int32),
                    np.array([-1, 0], np.int32), np.zeros(2, np.float32), 2)
    t = dtree.TreeBuffers(1, 1, 4, 2)
    upload_tree(t, 0, o)
    tg = torch.zeros((1, 2, 64), device="cuda")
    u = torch.rand((1, 2, 2), device="cuda")
    with pytest.raises(RuntimeError):
        dtree.verify(t, tg, uniforms=u, rule="iter_residual")  # needs the drafter rows
    with pytest.raises(RuntimeError):
        dtree.verify(t, tg, rule="target_match")  # needs uniforms
    out = dtree.verify(t, tg, uniforms=u, rule="target_match")  # no drafter rows needed
    torch.cuda.synchronize()
    assert int(out[1][0]) in (0, 1)
