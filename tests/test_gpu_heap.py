"""GPU parity of the heap mode (best-first heap with parent-conditioned edge
scores: exact sequential correction, TDES path scores) against the oracle.

The GPU selection gets the oracle's candidate tables (and, for the normalised
correction, the oracle's log-normalisers); the edge tables are computed on the
GPU from the same U, Vt or TDES weights.  Trees must match bit for bit,
scores included; the GPU's TDES table must equal the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from test_gpu_parity import f32, gen_logits, gpu_tree, oracle_tables, upload_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _same(g, o, what):
    assert g.n == o.n, (what, g.n, o.n)
    n = g.n
    for f in ("tok", "parent", "depth", "rank"):
        a, b = getattr(g, f)[:n], getattr(o, f)[:n]
        assert np.array_equal(a, b), (what, f, np.nonzero(a != b)[0][:10])
    assert np.array_equal(g.score[:n], o.score[:n]), (what, "score")


def _tdes(V, L, H, seed, device="cuda"):
    g = torch.Generator().manual_seed(seed)
    Ap = torch.randn((V, H), generator=g) * 0.3
    Ac = torch.randn((V, H), generator=g) * 0.3
    Dd = torch.randn((L, H), generator=g) * 0.3
    w = torch.randn(H, generator=g) * (1.0 / H ** 0.5)
    return Ap, Ac, Dd, w


def _run(batch, L, V, K, B, seed, term=None, root=True, dtype="bf16", norm=False, H=64, scale=3.0, p_spike=0.7):
    x = gen_logits(batch, L, V, dtype, scale, p_spike, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    rt = torch.randint(0, V, (batch,), generator=g, dtype=torch.int32) if root else None
    U = Vt = td = None
    R = 0
    if term == "markov":
        R = 64
        U = torch.randn((V, R), generator=g) * 0.1
        Vt = torch.randn((V, R), generator=g) * 0.1
    elif term == "tdes":
        Ap, Ac, Dd, w = _tdes(V, L, H, seed + 2)
        td = dtree.Tdes(Ap.cuda(), Ac.cuda(), Dd.cuda(), w.cuda(), b0=-0.1, s=0.8)
    p = dtree.Params(mode="heap", batch=batch, L=L, V=V, dtype=dtype, K=K, B=B, R=R,
                     U=U.cuda() if U is not None else None, Vt=Vt.cuda() if Vt is not None else None,
                     root_tok=rt.cuda() if root else None, markov_norm=norm, tdes=td)
    tree = dtree.TreeBuffers.for_params(p, max_nodes=B + 1)
    ws = dtree.make_workspace(p)
    tables, zs = {}, {}
    for b in range(batch):
        tables[b] = oracle_tables(x[b], K)
        upload_tables(tree, b, *tables[b])
    if norm:
        zv = dtree.znorm_view(p, ws)
        for b in range(batch):
            zs[b] = oracle.markov_norm(f32(x[b]), tables[b][1], U.numpy(), Vt.numpy(), int(rt[b]) if root else -1)
            zv[b].copy_(torch.from_numpy(zs[b]))
    dtree.select(p, tree, workspace=ws)
    torch.cuda.synchronize()
    assert int(tree.status.abs().sum()) == 0
    for b in range(batch):
        _, ids, lps = tables[b]
        r = int(rt[b]) if root else -1
        E = None
        if term == "markov":
            E = oracle.markov_table(ids, U.numpy(), Vt.numpy(), r)
        elif term == "tdes":
            E = oracle.tdes_table(ids, Ap.numpy(), Ac.numpy(), Dd.numpy(), w.numpy(), -0.1, 0.8, r)
            Eg = ws[0][:batch * L * K * K * 4].view(torch.float32).view(batch, L, K, K)[b].cpu().numpy()
            assert np.array_equal(Eg[1:], E[1:]), "TDES table"
            if root:  # without a root token the depth-1 row is not written
                assert np.array_equal(Eg[0, 0], E[0, 0]), "TDES root row"
        want = oracle.heap_select(lps, ids, B, E=E, znorm=zs.get(b))
        _same(gpu_tree(tree, b), want, (term, b))
    return p, tree, ws


@pytest.mark.parametrize("L,V,K,B,dtype,p_spike", [
    (4, 3000, 8, 40, "bf16", 0.7),     # every order row precomputed
    (6, 1000, 12, 200, "f32", 0.0),    # deep, many pops
    (16, 5000, 64, 64, "bf16", 0.7),   # rows beyond shared memory: computed on demand
    (3, 600, 4, 500, "bf16", 0.7),     # budget above the lattice size (4 + 16 + 64)
])
def test_heap_without_term_is_ddtree(L, V, K, B, dtype, p_spike):
    x = gen_logits(2, L, V, dtype, 3.0, p_spike, seed=L * V)
    if dtype == "bf16":  # coarse logits: many equal scores, ties broken by the descriptor
        x = (x.float() * 2).round().div(2).to(torch.bfloat16)
    p = dtree.Params(mode="heap", batch=2, L=L, V=V, dtype=dtype, K=K, B=B)
    tree = dtree.TreeBuffers.for_params(p, max_nodes=B + 1)
    tabs = {}
    for b in range(2):
        tabs[b] = oracle_tables(x[b], K)
        upload_tables(tree, b, *tabs[b])
    dtree.select(p, tree)
    torch.cuda.synchronize()
    for b in range(2):
        _same(gpu_tree(tree, b), oracle.ddtree(tabs[b][2], tabs[b][1], B), ("ddtree", b))


@pytest.mark.parametrize("root", [True, False])
@pytest.mark.parametrize("L,V,K,B", [(5, 4000, 8, 60), (16, 151936, 16, 512), (16, 20000, 64, 64)])
def test_heap_markov_term(root, L, V, K, B):
    _run(2, L, V, K, B, seed=K + B, term="markov", root=root)


@pytest.mark.parametrize("L,V,K,B", [(4, 3000, 8, 50), (16, 151936, 16, 512)])
def test_heap_normalised_markov_term(L, V, K, B):
    _run(2, L, V, K, B, seed=3 * K, term="markov", norm=True)


@pytest.mark.parametrize("root", [True, False])
@pytest.mark.parametrize("L,V,K,B,H", [(4, 2000, 8, 40, 32), (16, 151936, 16, 256, 256), (8, 9000, 32, 300, 100)])
def test_heap_tdes_term(root, L, V, K, B, H):
    _run(2, L, V, K, B, seed=H + K, term="tdes", root=root, H=H)


def test_heap_build_end_to_end_and_mask():
    # stage 1 on the GPU, then the heap with the TDES term; the mask from
    # dt_select_mask equals dt_tree_mask on the same tree
    batch, L, V, K, B = 4, 16, 151936, 16, 512
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=77)
    Ap, Ac, Dd, w = _tdes(V, L, 128, 78)
    p = dtree.Params(mode="heap", batch=batch, L=L, V=V, dtype="bf16", K=K, B=B,
                     tdes=dtree.Tdes(Ap.cuda(), Ac.cuda(), Dd.cuda(), w.cuda(), b0=0.2, s=1.0))
    tree = dtree.TreeBuffers.for_params(p, max_nodes=B + 1)
    ws = dtree.make_workspace(p)
    m1, p1 = dtree.alloc_mask(tree)
    m2, p2 = dtree.alloc_mask(tree)
    dtree.build_tree_mask(p, x.cuda(), tree, m1, p1, workspace=ws, pos_offset=5)
    dtree.tree_mask(tree, m2, p2, pos_offset=5)
    torch.cuda.synchronize()
    assert int(tree.status.abs().sum()) == 0
    assert torch.equal(m1, m2) and torch.equal(p1, p2)
    n = tree.n_nodes.cpu().numpy()
    assert np.all(n == B + 1)
    for b in range(batch):
        t = gpu_tree(tree, b)
        assert np.all(t.parent[1:] < np.arange(1, t.n))  # parents first
