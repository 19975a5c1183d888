"""DARTree with the full-vocabulary normalised correction, on the GPU.

dt_markov_norm computes the log-normaliser table on the tensor cores, each fp32
table split into a bf16 head and tail with all four products accumulated in
fp32; it is compared with the oracle's double-precision table within the bound
that split implies (include/dtree.h): the operand split leaves
2^-18 |U| + 2^-18 |Vt| + 2^-36 per product and the accumulator's sixteen fp32
accumulation steps at most 2^-19 of the magnitudes, so
|dz| <= 2^-16 * max_v sum_k |U[u][k] * Vt[v][k]| + 6e-6 (the second term: the
fp32 log-sum-exp over V and the stage-1 normaliser it subtracts).  Every
table entry must also lie within 1e-5 of the oracle's.  The normalised
selection is bit-exact when both sides get the same tables and normalisers,
and end to end (the GPU computing stage 1, the table and the selection from
raw logits) differs from the oracle's only by near-ties.  Inputs flow only
from the oracle to the GPU."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_bf16_gb300 import dtree
from test_gpu_parity import assert_same_tree, check_end_to_end, f32, gen_logits, gpu_tree, oracle_tables, upload_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _tables(V, R, seed):
    g = torch.Generator().manual_seed(seed)
    U = torch.randn((V, R), generator=g) * 0.1
    Vt = torch.randn((V, R), generator=g) * 0.1
    return U, Vt


Z_TOL = 1e-5  # every normaliser within this of the oracle's


def _bound(U, Vt, u):
    """2^-16 * max_v sum_k |U[u][k] * Vt[v][k]| + 6e-6 (the head/tail split and fp32 accumulation)."""
    a = np.abs(U[u].numpy().astype(np.float64))
    return min(2.0 ** -16 * float((np.abs(Vt.numpy().astype(np.float64)) @ a).max()) + 6e-6, Z_TOL)


def _setup(batch, L, V, K, seed, dtype="bf16", root=True):
    x = gen_logits(batch, L, V, dtype, 3.0, 0.7, seed=seed)
    U, Vt = _tables(V, 64, seed + 1)
    g = torch.Generator().manual_seed(seed + 2)
    rt = torch.randint(0, V, (batch,), generator=g, dtype=torch.int32) if root else None
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype=dtype, K=K, W=32, B=512, beta=-0.25, R=64,
                     U=U.cuda(), Vt=Vt.cuda(), root_tok=rt.cuda() if root else None, markov_norm=True)
    tree = dtree.TreeBuffers.for_params(p, max_nodes=min(512, 32 * L) + 1)
    tables = {}
    for b in range(batch):
        tables[b] = oracle_tables(x[b], K)
        upload_tables(tree, b, *tables[b])
    return x, U, Vt, rt, p, tree, tables


@pytest.mark.parametrize("batch,L,V,K,dtype,root", [
    (2, 4, 3000, 8, "bf16", True),    # several row tiles of 128, ragged vocabulary slices
    (1, 3, 1001, 5, "f32", False),    # fp32 logits, odd V (unaligned rows), no root token
    (3, 2, 260, 16, "bf16", True),    # vocabulary shorter than two MMA steps
])
def test_normaliser_table_matches_oracle(batch, L, V, K, dtype, root):
    x, U, Vt, rt, p, tree, tables = _setup(batch, L, V, K, seed=V + K, dtype=dtype, root=root)
    ws = dtree.make_workspace(p)
    dtree.markov_norm(p, x.cuda(), tree, ws)
    torch.cuda.synchronize()
    z = dtree.znorm_view(p, ws).cpu().numpy()
    for b in range(batch):
        want = oracle.markov_norm(f32(x[b]), tables[b][1], U.numpy(), Vt.numpy(), int(rt[b]) if root else -1)
        for d in range(L):
            for i in range(K):
                u = (int(rt[b]) if (root and i == 0) else -1) if d == 0 else int(tables[b][1][d - 1][i])
                if u < 0:
                    assert z[b, d, i] == 0.0
                    continue
                assert abs(float(z[b, d, i]) - float(want[d, i])) <= _bound(U, Vt, u), (b, d, i)


def test_normaliser_table_full_vocabulary_sampled_rows():
    batch, L, V, K = 2, 16, 151936, 16
    x, U, Vt, rt, p, tree, tables = _setup(batch, L, V, K, seed=7)
    ws = dtree.make_workspace(p)
    dtree.markov_norm(p, x.cuda(), tree, ws)
    torch.cuda.synchronize()
    z = dtree.znorm_view(p, ws).cpu().numpy()
    rng = np.random.default_rng(0)
    for b in range(batch):
        rows = [0] + [int(r) for r in rng.choice(np.arange(K, L * K), 4, replace=False)]
        for r in rows:
            d, i = divmod(r, K)
            want = oracle.markov_norm(f32(x[b]), tables[b][1], U.numpy(), Vt.numpy(), int(rt[b]), only_row=r)
            u = int(rt[b]) if d == 0 else int(tables[b][1][d - 1][i])
            assert abs(float(z[b, d, i]) - float(want[d, i])) <= _bound(U, Vt, u), (b, d, i)


@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_normalised_selection_is_bit_exact(beta):
    batch, L, V, K = 2, 6, 2000, 8
    x, U, Vt, rt, p, tree, tables = _setup(batch, L, V, K, seed=31)
    p.beta = beta
    p.B = 60
    p.W = 12
    tree = dtree.TreeBuffers.for_params(p, max_nodes=61)
    for b in range(batch):
        upload_tables(tree, b, *tables[b])
    ws = dtree.make_workspace(p)
    zv = dtree.znorm_view(p, ws)
    want = {}
    for b in range(batch):
        z = oracle.markov_norm(f32(x[b]), tables[b][1], U.numpy(), Vt.numpy(), int(rt[b]))
        zv[b].copy_(torch.from_numpy(z))
        t, info, _ = oracle.dartree(tables[b][2], tables[b][1], U.numpy(), Vt.numpy(), int(rt[b]), W=12, beta=beta,
                                    B=60, Mmax=61, znorm=z)
        assert info["violations"] == 0  # q~ <= 1: Lemma 1's hypothesis holds
        want[b] = t.trimmed()
    dtree.select(p, tree, workspace=ws)
    torch.cuda.synchronize()
    for b in range(batch):
        assert_same_tree(gpu_tree(tree, b), want[b], "normalised dartree b=%d" % b)
    assert int(tree.status.abs().sum()) == 0


def test_build_tree_with_normalisation_end_to_end():
    # the DARTree workload shape: stage 1, normalisers and selection on the GPU
    batch, L, V, K = 8, 16, 151936, 16
    x = gen_logits(batch, L, V, "bf16", 3.0, 0.7, seed=5)
    U, Vt = _tables(V, 64, 6)
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype="bf16", K=K, W=32, B=512, beta=0.0, R=64,
                     U=U.cuda(), Vt=Vt.cuda(), markov_norm=True)
    tree = dtree.TreeBuffers.for_params(p, max_nodes=min(512, 32 * L) + 1)
    ws = dtree.make_workspace(p)
    dtree.build_tree(p, x.cuda(), tree, workspace=ws)
    torch.cuda.synchronize()
    assert int(tree.status.abs().sum()) == 0  # no violation, no best-first fallback, no timeout
    z = dtree.znorm_view(p, ws).cpu().numpy()
    assert np.all(np.isfinite(z)) and np.all(z[:, 0, :] == 0.0)  # no root token: no term at position 0
    n = tree.n_nodes.cpu().numpy()
    assert np.all(n == 497)  # |S| = 16 + 15 * 32 < B: the whole supertree
    for b in range(batch):
        t = gpu_tree(tree, b)
        assert np.all(t.score[1:] <= 0.0)  # normalised log-probabilities only decrease along a path
        assert np.all(np.diff(t.score[1:]) <= 0.0)
    # against the oracle from the same raw logits: its own stage 1, normaliser table and selection
    for b in (0, 5):
        _, ids, lps = oracle_tables(x[b], K)
        zo = oracle.markov_norm(f32(x[b]), ids, U.numpy(), Vt.numpy(), -1)
        err = np.abs(z[b].astype(np.float64) - zo)
        assert err.max() < Z_TOL, err.max()
        ot, info, _ = oracle.dartree(lps, ids, U.numpy(), Vt.numpy(), -1, 32, 0.0, 512, Mmax=tree.max_nodes, znorm=zo)
        assert info["violations"] == 0
        E = oracle.markov_table(ids, U.numpy(), Vt.numpy(), -1)
        check_end_to_end(gpu_tree(tree, b), ot.trimmed(), lps, "dartree", E=E, znorm=zo, beta=0.0, eps_z=Z_TOL,
                         what="normalised dartree b=%d (max normaliser error %.1e)" % (b, err.max()))
