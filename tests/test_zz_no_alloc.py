"""dt_select_dartree_noalloc against dt_select, through the C ABI.

Some callers cannot allocate device memory -- a serving framework that owns
the whole device budget, or a latency-critical loop where cudaMalloc is not
allowed because it can synchronise the device -- so they cannot pass the
DARTree workspace.  The allocation-free entry point keeps that table in a fixed
array inside the library instead.  Its trees must equal the workspace entry
point's, bit for bit, on two calls in a row on one shape with different
inputs: the second call finds the first call's table in the shared array at
the same offsets.  With a root token a call also uses the depth-1 entries,
without one it skips them, so both orders are run: a call with root tokens
after one without (it must write what it reads), and the reverse (it must not
read the stale depth-1 entries).  This file is collected last."""
import ctypes

import pytest
import torch

from speculative_decoding_draft_bf16_gb300 import dtree

pytestmark = pytest.mark.gpu

FIELDS = ("node_tok", "parent", "depth", "rank", "n_nodes", "status")


def _case(seed, batch, L, V, K, W, B, R, root):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((batch, L, V), generator=g) * 3).to(torch.bfloat16)
    U = torch.randn((V, R), generator=g) * 0.1
    Vt = torch.randn((V, R), generator=g) * 0.1
    rt = torch.randint(0, V, (batch,), generator=g, dtype=torch.int32) if root else None
    p = dtree.Params(mode="dartree", batch=batch, L=L, V=V, dtype="bf16", K=K, W=W, B=B, beta=-0.25, R=R,
                     U=U.cuda(), Vt=Vt.cuda(), root_tok=rt.cuda() if root else None)
    return x.cuda(), p, min(B, W * L) + 1


def _check_one(seed, shape, root):
    batch, L, V, K, W, B, R = shape
    x, p, max_nodes = _case(seed, batch, L, V, K, W, B, R, root)
    ref = dtree.TreeBuffers.for_params(p, max_nodes=max_nodes)
    got = dtree.TreeBuffers.for_params(p, max_nodes=max_nodes)
    dtree.candidates(p, x, ref)
    for f in ("lse", "cand_id", "cand_lp"):
        getattr(got, f).copy_(getattr(ref, f))
    dtree.select(p, ref, workspace=dtree.make_workspace(p))
    dtree.select_dartree_noalloc(p, got)
    torch.cuda.synchronize()
    for f in FIELDS:
        assert torch.equal(getattr(ref, f), getattr(got, f)), (seed, root, f)
    assert torch.equal(ref.score.view(torch.int32), got.score.view(torch.int32)), (seed, root)


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_lib):
    shapes = [
        (3, 6, 2000, 8, 6, 20, 16),          # small
        (8, 16, 151936, 16, 32, 512, 64),    # the batch-8 supertree workload shape
    ]
    for i, shape in enumerate(shapes):
        first_root = i % 2 == 0               # small: root tokens first; large: none first
        _check_one(11 + 2 * i, shape, first_root)
        _check_one(12 + 2 * i, shape, not first_root)


def test_noalloc_rejects_tables_beyond_the_fixed_size(cuda_lib):
    V, R = 1000, 8
    U = torch.zeros((V, R), device="cuda")
    # 64 * 16 * 64 * 64 floats = 16 MiB > DT_NOALLOC_TABLE_BYTES (4 MiB)
    p = dtree.Params(mode="dartree", batch=64, L=16, V=V, dtype="bf16", K=64, W=8, B=64, R=R, U=U, Vt=U)
    tree = dtree.TreeBuffers.for_params(p, max_nodes=65)
    rc = cuda_lib.dt_select_dartree_noalloc(ctypes.byref(p.struct()), ctypes.byref(tree.struct()), None)
    assert rc == -2  # DT_ERR_UNSUPPORTED
    # another mode is not this entry point's job
    q = dtree.Params(mode="ddtree", batch=1, L=4, V=V, dtype="bf16", K=4, B=8)
    t2 = dtree.TreeBuffers.for_params(q)
    assert cuda_lib.dt_select_dartree_noalloc(ctypes.byref(q.struct()), ctypes.byref(t2.struct()), None) == -1
