"""CPU checks of the C ABI: the library loads without a GPU, exports every
function include/dtree.h declares, and rejects invalid arguments on the host
before anything touches CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from speculative_decoding_draft_bf16_gb300 import dtree

HEADER = os.path.join(ROOT, "include", "dtree.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dt_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dt_candidates", "dt_select", "dt_build_tree", "dt_tree_mask", "dt_verify", "dt_workspace_size",
              "dt_status_str", "dt_version"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = dtree.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_static_strings_and_version():
    L = dtree.lib()
    assert L.dt_version() >= 100
    assert L.dt_status_str(0) == b"ok"
    assert L.dt_status_str(-1) == b"invalid argument"
    assert L.dt_status_str(-4).startswith(b"CUDA")


def _params(**kw):
    base = dict(mode="ddtree", batch=1, L=4, V=32, dtype="f32", K=4, B=8)
    base.update(kw)
    return dtree.Params(**base)


class _FakeTree:
    """A dt_tree with non-NULL fake device pointers: host validation never
    dereferences them, and every case below fails validation first."""

    def __init__(self, batch, L, Kc, max_nodes):
        self.batch, self.L, self.Kc, self.max_nodes = batch, L, Kc, max_nodes

    def struct(self):
        p = [ctypes.c_void_p(0x1000 + 16 * i) for i in range(10)]
        return dtree.TreeStruct(self.max_nodes, self.Kc, self.L, *p)


def _call_build(p, tree, logits_ptr=0x2000):
    return dtree.lib().dt_build_tree(ctypes.byref(p.struct()), ctypes.c_void_p(logits_ptr),
                                     ctypes.byref(tree.struct()), None, 0, None)


@pytest.mark.parametrize("bad", [
    dict(batch=0), dict(L=0), dict(L=33), dict(V=0), dict(K=0), dict(K=33), dict(B=0), dict(B=1025),
    dict(mode="talon", N=0, talon_k=1, mu=0.5), dict(mode="talon", N=10, talon_k=11, mu=0.5),
    dict(mode="dartree", W=0, K=4, B=8), dict(mode="dartree", W=4, K=4, B=8, beta=0.5),
    dict(mode="dartree", W=2000, K=4, B=8),
])
def test_build_rejects_invalid_params(bad):
    p = _params(**bad)
    Kc = p.Kc if p.Kc > 0 else 1
    tree = _FakeTree(max(p.batch, 1), max(p.L, 1), Kc, max(min(p.budget + 1, 1025), 1))
    assert _call_build(p, tree) == -1


def test_build_rejects_mismatched_tree_and_null_pointers():
    p = _params()
    assert _call_build(p, _FakeTree(1, 4, 5, 9)) == -1      # Kc != K
    assert _call_build(p, _FakeTree(1, 3, 4, 9)) == -1      # L mismatch
    assert _call_build(p, _FakeTree(1, 4, 4, 8)) == -1      # max_nodes < B + 1
    assert _call_build(p, _FakeTree(1, 4, 4, 9), logits_ptr=0) == -1  # NULL logits
    L = dtree.lib()
    assert L.dt_build_tree(None, None, None, None, 0, None) == -1


def test_unsupported_sizes():
    p = _params(V=16 * 32768 + 1, K=4)
    assert _call_build(p, _FakeTree(1, 4, 4, 9)) == -2


def test_mask_and_verify_reject_invalid_arguments():
    L = dtree.lib()
    t = _FakeTree(1, 4, 4, 9).struct()
    fake = ctypes.c_void_p(0x3000)
    assert L.dt_tree_mask(ctypes.byref(t), 0, 0, fake, fake, None) == -1
    assert L.dt_tree_mask(ctypes.byref(t), 1, 0, None, fake, None) == -1
    t_big = _FakeTree(1, 4, 4, 1026).struct()
    assert L.dt_tree_mask(ctypes.byref(t_big), 1, 0, fake, fake, None) == -1
    # verify: temperature other than 0/1, NULL target, T=1 without uniforms
    args = lambda temp, tgt, drf, uni: L.dt_verify(ctypes.byref(t), 1, 32, 1, tgt, None, drf, ctypes.c_float(temp),
                                                   uni, fake, fake, fake, None, None)
    assert args(0.5, fake, fake, fake) == -2
    assert args(0.0, None, None, None) == -1
    assert args(1.0, fake, None, fake) == -1
    assert args(1.0, fake, fake, None) == -1
    # verify with an explicit rule: unknown rules; the drafter rows are needed by
    # the ratio and residual rules, uniforms by every T=1 rule
    rule = lambda r, tgt, drf, uni: L.dt_verify_rule(ctypes.byref(t), 1, 32, 1, tgt, None, drf, r, uni, fake, fake,
                                                     fake, None, None)
    assert rule(-1, fake, fake, fake) == -1 and rule(4, fake, fake, fake) == -1
    for r in (dtree.VERIFY_RULES["ratio"], dtree.VERIFY_RULES["iter_residual"]):
        assert rule(r, fake, None, fake) == -1
        assert rule(r, fake, fake, None) == -1
    assert rule(dtree.VERIFY_RULES["target_match"], fake, fake, None) == -1
    assert rule(dtree.VERIFY_RULES["greedy"], None, None, None) == -1


def test_workspace_size():
    assert dtree.workspace_size(_params()) == 0
    assert dtree.workspace_size(_params(mode="talon", N=60, talon_k=10, mu=0.03)) == 0
    # DARTree with a Markov term: batch * L * K * K * 4 bytes
    import torch
    U = torch.zeros((32, 8))
    p = _params(mode="dartree", batch=3, L=4, K=4, W=4, B=8, R=8)
    p.U = U
    p.Vt = U
    assert dtree.workspace_size(p) == 3 * 4 * 4 * 4 * 4


def test_stage1_plan_picks_the_kernel_by_rows_and_list_length():
    # many rows, or long candidate lists: a CTA per row (no device query needed)
    p = dtree.Params(mode="ddtree", batch=64, L=16, V=151936, dtype="bf16", K=60, B=60)
    assert dtree.stage1_plan(p) == ("rows", 1)
    p = dtree.Params(mode="talon", batch=1, L=16, V=151936, dtype="bf16", talon_k=10, mu=0.03, N=1024)
    assert dtree.stage1_plan(p) == ("rows", 1)
    # one request: each row over a cluster (a power of two, chunks of at most 32768 elements)
    p = dtree.Params(mode="ddtree", batch=1, L=16, V=151936, dtype="bf16", K=256, B=256)
    kind, s = dtree.stage1_plan(p)
    assert kind == "cluster" and s in (8, 16)
    with pytest.raises(dtree.DtError):
        dtree.stage1_plan(dtree.Params(mode="ddtree", batch=1, L=16, V=100, dtype="bf16", K=101, B=4))
    L = dtree.lib()
    k = ctypes.c_int32()
    assert L.dt_stage1_plan(None, ctypes.byref(k), ctypes.byref(k)) == -1
    assert L.dt_stage1_ceiling(None, None, None, None, None) == -1


def test_fused_entry_points_and_normalisation_reject_invalid_arguments():
    L = dtree.lib()
    fake = ctypes.c_void_p(0x3000)
    good = dtree.Params(mode="ddtree", batch=1, L=4, V=32, dtype="bf16", K=4, B=8)
    bad = dtree.Params(mode="ddtree", batch=0, L=4, V=32, dtype="bf16", K=4, B=8)
    t = _FakeTree(1, 4, 4, 9).struct()
    # null mask / positions, invalid parameters: rejected on the host
    assert L.dt_select_mask(ctypes.byref(good.struct()), ctypes.byref(t), None, 0, 0, None, fake, None) == -1
    assert L.dt_select_mask(ctypes.byref(bad.struct()), ctypes.byref(t), None, 0, 0, fake, fake, None) == -1
    assert L.dt_build_tree_mask(ctypes.byref(bad.struct()), fake, ctypes.byref(t), None, 0, 0, fake, fake,
                                None) == -1
    assert L.dt_build_tree_mask(ctypes.byref(good.struct()), fake, ctypes.byref(t), None, 0, 0, fake, None,
                                None) == -1
    # the normalised DARTree correction: needs a Markov table of rank 64 and 16-byte aligned tables
    def dart(**kw):
        q = dict(mode="dartree", batch=1, L=4, V=32, dtype="bf16", K=4, W=4, B=8, R=64, markov_norm=True)
        q.update(kw)
        return dtree.Params(**q)
    U = ctypes.c_void_p(0x10000)

    def with_tables(q, u=U, r=None):
        st = q.struct()
        st.U, st.Vt = u, U
        st.R = q.R if r is None else r
        return st
    s = with_tables(dart())
    td = _FakeTree(1, 4, 4, 9).struct()
    w = ctypes.c_int(0)
    assert L.dt_workspace_size(ctypes.byref(s), ctypes.byref(w)) > 0 and w.value == 1
    s32 = with_tables(dart(R=32))
    assert L.dt_markov_norm(ctypes.byref(s32), fake, ctypes.byref(td), fake, 1 << 30, None) == -2
    s_unaligned = with_tables(dart(), u=ctypes.c_void_p(0x10004))
    assert L.dt_markov_norm(ctypes.byref(s_unaligned), fake, ctypes.byref(td), fake, 1 << 30, None) == -1
    s_noterm = dart(R=0).struct()
    assert L.dt_markov_norm(ctypes.byref(s_noterm), fake, ctypes.byref(td), fake, 1 << 30, None) == -1
    # the allocation-free selection does not take the normalised correction
    assert L.dt_select_dartree_noalloc(ctypes.byref(s), ctypes.byref(td), None) == -2


def test_heap_mode_rejects_invalid_arguments():
    L = dtree.lib()
    t = _FakeTree(1, 4, 4, 9).struct()
    fake = ctypes.c_void_p(0x3000)
    heap = dtree.Params(mode="heap", batch=1, L=4, V=32, dtype="bf16", K=4, B=8)
    # no edge term: no workspace
    w = ctypes.c_int(0)
    assert L.dt_workspace_size(ctypes.byref(heap.struct()), ctypes.byref(w)) == 0 and w.value == 1
    # a TDES scorer: an edge table of batch * L * K * K floats, rounded to 256 bytes
    st = heap.struct()
    tds = dtree.TdesStruct(8, fake, fake, fake, fake, 0.0, 1.0)
    st.tdes = ctypes.pointer(tds)
    assert L.dt_workspace_size(ctypes.byref(st), ctypes.byref(w)) == 256 and w.value == 1
    assert L.dt_select(ctypes.byref(st), ctypes.byref(t), None, 0, None) == -1  # workspace missing
    for bad in (dtree.TdesStruct(0, fake, fake, fake, fake, 0.0, 1.0),
                dtree.TdesStruct(8, None, fake, fake, fake, 0.0, 1.0),
                dtree.TdesStruct(8, fake, fake, fake, None, 0.0, 1.0)):
        st.tdes = ctypes.pointer(bad)
        assert L.dt_select(ctypes.byref(st), ctypes.byref(t), fake, 1 << 20, None) == -1
    # the normaliser belongs to the Markov term, not to TDES
    st.tdes = ctypes.pointer(tds)
    st.markov_norm = 1
    assert L.dt_select(ctypes.byref(st), ctypes.byref(t), fake, 1 << 20, None) == -1
    # candidate lists longer than 256
    big = dtree.Params(mode="heap", batch=1, L=4, V=1000, dtype="bf16", K=300, B=8)
    assert L.dt_select(ctypes.byref(big.struct()), ctypes.byref(_FakeTree(1, 4, 300, 9).struct()), None, 0,
                       None) == -2


def test_budget_policies_reject_invalid_arguments():
    L = dtree.lib()
    fake = ctypes.c_void_p(0x3000)
    t = _FakeTree(2, 4, 4, 9).struct()
    # uniform per-depth budgets are DARTree's; per-request budgets are DDTree's and the heap's
    bad = [dtree.Params(mode="ddtree", batch=2, L=4, V=32, dtype="bf16", K=4, B=8, budget_policy="uniform")]
    st = dtree.Params(mode="dartree", batch=2, L=4, V=32, dtype="bf16", K=4, W=2, B=8).struct()
    st.budget = fake
    st2 = dtree.Params(mode="dartree", batch=2, L=4, V=32, dtype="bf16", K=4, W=2, B=3,
                       budget_policy="uniform").struct()  # B < L
    st3 = dtree.Params(mode="ddtree", batch=2, L=4, V=32, dtype="bf16", K=4, B=8).struct()
    st3.budget_policy = 7
    for s in [b.struct() for b in bad] + [st, st2, st3]:
        assert L.dt_select(ctypes.byref(s), ctypes.byref(t), None, 0, None) == -1
    # SABA parameters
    tr = _FakeTree(2, 4, 4, 9).struct()
    for q in (dtree.SabaStruct(0, 1.0, 1.0, 1, 8), dtree.SabaStruct(4, 0.0, 1.0, 1, 8),
              dtree.SabaStruct(4, 1.0, -1.0, 1, 8), dtree.SabaStruct(4, 1.0, 1.0, 0, 8),
              dtree.SabaStruct(4, 1.0, 1.0, 9, 8), dtree.SabaStruct(4, 1.0, 1.0, 1, 2000)):
        assert L.dt_saba_budget(ctypes.byref(q), ctypes.byref(tr), 2, None, 0, None, fake, fake, fake, fake,
                                None) == -1
    ok = dtree.SabaStruct(4, 1.0, 1.0, 1, 8)
    assert L.dt_saba_budget(ctypes.byref(ok), ctypes.byref(tr), 2, None, 0, None, None, fake, fake, fake, None) == -1
    assert L.dt_saba_budget(ctypes.byref(ok), ctypes.byref(tr), 2, fake, 0, None, fake, fake, fake, fake, None) == -1


def test_verify_markov_rejects_invalid_arguments():
    L = dtree.lib()
    fake = ctypes.c_void_p(0x3000)
    t = _FakeTree(1, 4, 4, 9).struct()

    def params(R=64, vt=0x10000, K=4):
        q = dtree.Params(mode="dartree", batch=1, L=4, V=32, dtype="bf16", K=K, W=4, B=8).struct()
        q.R, q.U, q.Vt = R, ctypes.c_void_p(0x20000), ctypes.c_void_p(vt)
        return q
    call = lambda q, z=fake: L.dt_verify_markov(ctypes.byref(q), ctypes.byref(t), fake, None, fake, z, fake, fake,
                                                fake, fake, None, None)
    assert call(params(), z=None) == -1        # no normalisers
    assert call(params(R=66)) == -1            # more than 64 columns
    assert call(params(R=62)) == -1            # not a multiple of 4
    assert call(params(vt=0x10004)) == -1      # Vt not 16-byte aligned
    assert call(params(K=5)) == -1             # tree lists of another length


def test_binding_size_checks_reject_short_buffers_and_small_trees():
    # the C ABI takes bare pointers: the binding compares sizes before any launch
    import torch
    dtree._need_numel(torch.zeros(12), 12, "x")
    with pytest.raises(ValueError):
        dtree._need_numel(torch.zeros(11), 12, "x")
    t = _FakeTree(2, 4, 4, 9)
    dtree._need_batch(t, 2)
    with pytest.raises(ValueError):
        dtree._need_batch(t, 3)
    with pytest.raises(ValueError):
        dtree._need(torch.zeros(4), name="cpu tensor")  # a host tensor never reaches a kernel
