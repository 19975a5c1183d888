"""GPU parity of the T=1 walk against the normalised DARTree proposal
(dt_verify_markov): the oracle's DARTree trees, log-normalisers, target rows and
uniforms go to the GPU; accepted paths and emitted tokens must match the
oracle's or_verify_t1_markov bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from test_gpu_parity import f32, gen_logits, oracle_tables, row_lse, verify_tree_buffers

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _case(batch, L, V, K, W, B, dtype, seed, root=True, zero_U=False):
    x = gen_logits(batch, L, V, dtype, 2.0, 0.7, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    U = torch.randn((V, 64), generator=g) * 0.1
    Vt = torch.randn((V, 64), generator=g) * 0.1
    if zero_U:
        U.zero_()
    rt = torch.randint(0, V, (batch,), generator=g, dtype=torch.int32) if root else None
    otrees, dl, zs = [], [], []
    for b in range(batch):
        l32, ids, lps = oracle_tables(x[b], K)
        r = int(rt[b]) if root else -1
        z = oracle.markov_norm(f32(x[b]), ids, U.numpy(), Vt.numpy(), r)
        t, _, _ = oracle.dartree(lps, ids, U.numpy(), Vt.numpy(), r, W, 0.0, B, znorm=z)
        otrees.append(t.trimmed())
        dl.append(l32)
        zs.append(z)
    Mmax = min(B, W * L) + 1
    tree = verify_tree_buffers(otrees, L, K, Mmax, lse_rows=dl)
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype=dtype, K=K, W=W, B=B, R=64, U=U.cuda(),
                     Vt=Vt.cuda(), root_tok=rt.cuda() if root else None, markov_norm=True)
    return x, U, Vt, rt, otrees, dl, np.stack(zs), tree, p, Mmax


@pytest.mark.parametrize("dtype,V,root", [("f32", 3000, True), ("bf16", 10001, True), ("bf16", 4000, False)])
def test_markov_walk_matches_oracle(dtype, V, root):
    batch, L, K, W, B = 3, 6, 8, 6, 30
    x, U, Vt, rt, otrees, dl, z, tree, p, Mmax = _case(batch, L, V, K, W, B, dtype, seed=V, root=root)
    g = torch.Generator().manual_seed(V + 7)
    for mode in ("accept", "reject", "mixed"):
        tg = torch.zeros((batch, Mmax, V))
        for b, o in enumerate(otrees):
            for n in range(o.n):
                xd = x[b, min(int(o.depth[n]), L - 1)].float()
                tg[b, n] = xd if mode == "accept" else (-xd if mode == "reject" else torch.randn(V, generator=g) * 2)
        tg = tg.to(x.dtype)
        u = torch.rand((batch, 2, Mmax), generator=g)
        tl = np.stack([row_lse(f32(tg[b])) for b in range(batch)])
        for own in (False, True):
            out = dtree.verify_markov(p, tree, tg.cuda(), x.cuda(), torch.from_numpy(z).cuda(), u.cuda(),
                                      target_lse=None if own else torch.from_numpy(tl).cuda())
            torch.cuda.synchronize()
            for b in range(batch):
                acc, alen, nxt = oracle.verify_t1_markov(otrees[b], f32(tg[b]), f32(x[b]), dl[b], U.numpy(),
                                                         Vt.numpy(), int(rt[b]) if root else -1, z[b], u[b].numpy(),
                                                         L, Mmax, lse_in=None if own else tl[b])
                assert out[0][b].cpu().tolist() == acc.tolist(), (mode, own, b)
                assert int(out[1][b]) == alen and int(out[2][b]) == nxt, (mode, own, b)


def test_markov_walk_full_vocabulary():
    batch, L, V, K, W, B = 2, 16, 151936, 16, 32, 512
    x, U, Vt, rt, otrees, dl, z, tree, p, Mmax = _case(batch, L, V, K, W, B, "bf16", seed=3)
    g = torch.Generator().manual_seed(4)
    tg = torch.zeros((batch, Mmax, V))
    for b, o in enumerate(otrees):
        for n in range(o.n):
            xd = x[b, min(int(o.depth[n]), L - 1)].float()
            tg[b, n] = xd + torch.randn(V, generator=g) * 0.5  # close to the drafter: long walks, then a residual
    tg = tg.to(torch.bfloat16)
    u = torch.rand((batch, 2, Mmax), generator=g)
    tl = np.stack([row_lse(f32(tg[b])) for b in range(batch)])
    out = dtree.verify_markov(p, tree, tg.cuda(), x.cuda(), torch.from_numpy(z).cuda(), u.cuda(),
                              target_lse=torch.from_numpy(tl).cuda())
    torch.cuda.synchronize()
    for b in range(batch):
        acc, alen, nxt = oracle.verify_t1_markov(otrees[b], f32(tg[b]), f32(x[b]), dl[b], U.numpy(), Vt.numpy(),
                                                 int(rt[b]), z[b], u[b].numpy(), L, Mmax, lse_in=tl[b])
        assert out[0][b].cpu().tolist() == acc.tolist() and int(out[1][b]) == alen and int(out[2][b]) == nxt, b


def test_markov_walk_without_term_is_the_ratio_walk():
    batch, L, V, K, W, B = 2, 5, 2000, 6, 6, 25
    x, U, Vt, rt, otrees, dl, z, tree, p, Mmax = _case(batch, L, V, K, W, B, "f32", seed=11, zero_U=True)
    z[:] = 0.0
    tg = torch.randn((batch, Mmax, V), generator=torch.Generator().manual_seed(12)) * 2
    u = torch.rand((batch, 2, Mmax), generator=torch.Generator().manual_seed(13))
    a = dtree.verify_markov(p, tree, tg.cuda(), x.cuda(), torch.from_numpy(z).cuda(), u.cuda())
    b2 = dtree.verify(tree, tg.cuda(), draft=x.cuda(), uniforms=u.cuda(), rule="ratio")
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(a[i], b2[i])
