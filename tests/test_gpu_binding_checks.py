"""The binding refuses buffers the kernels would over-run, before any launch:
the C ABI sees bare pointers, so tensor sizes and the tree's request count are
checked in Python (a ValueError or TypeError, nothing enqueued)."""
import pytest
import torch

from speculative_decoding_draft_bf16_gb300 import dtree

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def test_short_or_mismatched_buffers_are_refused():
    p = dtree.Params(mode="ddtree", batch=2, L=4, V=64, dtype="bf16", K=4, B=8)
    tree = dtree.TreeBuffers.for_params(p)
    x = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):  # one request's logits for a two-request call
        dtree.build_tree(p, x[:1], tree)
    with pytest.raises(TypeError):  # fp32 logits for a bf16 parameter block
        dtree.build_tree(p, x.float(), tree)
    with pytest.raises(ValueError):  # rows of another vocabulary size
        dtree.build_tree(p, torch.zeros((2, 8, 32), dtype=torch.bfloat16, device="cuda"), tree)
    small = dtree.TreeBuffers(1, 4, 4, 9)
    with pytest.raises(ValueError):  # tree buffers for fewer requests than the call covers
        dtree.build_tree(p, x, small)
    with pytest.raises(ValueError):  # target rows for fewer nodes than max_nodes
        dtree.verify(tree, torch.zeros((2, 4, 64), device="cuda"))
    with pytest.raises(ValueError):  # uniforms for one request
        dtree.verify(tree, torch.zeros((2, 9, 64), dtype=torch.bfloat16, device="cuda"), temperature=1.0, draft=x,
                     uniforms=torch.zeros((1, 2, 9), device="cuda"))
    with pytest.raises(TypeError):  # bf16 drafter rows beside fp32 target rows: one element type is read
        dtree.verify(tree, torch.zeros((2, 9, 64), device="cuda"), temperature=1.0, draft=x,
                     uniforms=torch.zeros((2, 2, 9), device="cuda"))
    with pytest.raises(TypeError):  # the reverse: fp32 drafter rows beside bf16 target rows
        dtree.verify(tree, torch.zeros((2, 9, 64), dtype=torch.bfloat16, device="cuda"), temperature=1.0,
                     draft=x.float(), uniforms=torch.zeros((2, 2, 9), device="cuda"))
    pm = dtree.Params(mode="dartree", batch=2, L=4, V=64, dtype="bf16", K=4, W=4, B=8, R=2,
                      U=torch.zeros((64, 2), device="cuda"), Vt=torch.zeros((64, 2), device="cuda"),
                      markov_norm=True)
    with pytest.raises(TypeError):  # fp32 target rows for a bf16 parameter block (normalised DARTree walk)
        dtree.verify_markov(pm, tree, torch.zeros((2, 9, 64), device="cuda"), x,
                            torch.zeros((2, 4, 4), device="cuda"), torch.zeros((2, 2, 9), device="cuda"))
    mask, pos = dtree.alloc_mask(small)
    with pytest.raises(ValueError):  # a mask for one request
        dtree.select_mask(p, tree, mask, pos)
    with pytest.raises(ValueError):  # per-request budgets for one request
        q = dtree.Params(mode="ddtree", batch=2, L=4, V=64, dtype="bf16", K=4, B=8,
                         budgets=torch.ones(1, dtype=torch.int32, device="cuda"))
        dtree.select(q, tree)
    assert int(tree.n_nodes.sum()) == 0  # nothing ran
