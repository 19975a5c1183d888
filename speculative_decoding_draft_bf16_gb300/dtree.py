"""Python binding of the draft-tree C ABI (include/dtree.h).

Argument marshalling only: every step of build, mask and verify runs in the
CUDA kernels of libdtree.so.  Tensors must be CUDA tensors, contiguous, of the
documented dtype; the library writes into caller-owned buffers on the current
torch stream (or the stream given).  A missing or unloadable library raises --
there is no other code path.
"""
import ctypes
import dataclasses
import math
import os

import torch

from . import build as _build

DT_MODE = {"ddtree": 0, "dartree": 1, "talon": 2, "heap": 3}
BUDGET_POLICY = {"topb": 0, "uniform": 1}
DT_BF16, DT_F32 = 0, 1
DT_DEV_BAD_TREE, DT_DEV_TIMEOUT, DT_DEV_BESTFIRST = 0x1, 0x2, 0x4
DT_DEV_VIOLATION_SHIFT = 8
DT_STAGE1_CLUSTER, DT_STAGE1_ROWS = 1, 2
# acceptance rules of dt_verify_rule
VERIFY_RULES = {"greedy": 0, "ratio": 1, "iter_residual": 2, "target_match": 3}
MAX_NODES = 1025
MAX_KC = 1024

_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class TdesStruct(ctypes.Structure):
    _fields_ = [("H", _i32), ("Ap", _vp), ("Ac", _vp), ("Dd", _vp), ("w", _vp), ("b0", ctypes.c_float),
                ("s", ctypes.c_float)]


class BuildParams(ctypes.Structure):
    _fields_ = [("mode", _i32), ("batch", _i32), ("L", _i32), ("V", _i32), ("dtype", _i32),
                ("K", _i32), ("B", _i32), ("W", _i32), ("beta", ctypes.c_float), ("R", _i32),
                ("U", _vp), ("Vt", _vp), ("root_tok", _vp), ("talon_k", _i32),
                ("log_mu", ctypes.c_float), ("N", _i32), ("markov_norm", _i32),
                ("tdes", ctypes.POINTER(TdesStruct)), ("budget_policy", _i32), ("budget", _vp)]


class SabaStruct(ctypes.Structure):
    _fields_ = [("window", _i32), ("c_verify", ctypes.c_float), ("c_fixed", ctypes.c_float), ("B_min", _i32),
                ("B_max", _i32)]


class TreeStruct(ctypes.Structure):
    _fields_ = [("max_nodes", _i32), ("Kc", _i32), ("L", _i32), ("node_tok", _vp), ("parent", _vp),
                ("depth", _vp), ("rank", _vp), ("score", _vp), ("n_nodes", _vp), ("lse", _vp),
                ("cand_id", _vp), ("cand_lp", _vp), ("status", _vp)]


_LIB = None


def lib():
    """Load libdtree.so (compiling it first if it has never been built)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            path = _build.build()
        L = ctypes.CDLL(path)
        bp = ctypes.POINTER(BuildParams)
        tp = ctypes.POINTER(TreeStruct)
        L.dt_workspace_size.restype = ctypes.c_size_t
        L.dt_workspace_size.argtypes = [bp, ctypes.POINTER(ctypes.c_int)]
        L.dt_candidates.restype = _i32
        L.dt_candidates.argtypes = [bp, _vp, tp, _vp]
        L.dt_markov_norm.restype = _i32
        L.dt_markov_norm.argtypes = [bp, _vp, tp, _vp, ctypes.c_size_t, _vp]
        L.dt_stage1_plan.restype = _i32
        L.dt_stage1_plan.argtypes = [bp, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
        L.dt_stage1_ceiling.restype = _i32
        L.dt_stage1_ceiling.argtypes = [bp, _vp, _vp, _vp, _vp]
        L.dt_select.restype = _i32
        L.dt_select.argtypes = [bp, tp, _vp, ctypes.c_size_t, _vp]
        L.dt_build_tree.restype = _i32
        L.dt_build_tree.argtypes = [bp, _vp, tp, _vp, ctypes.c_size_t, _vp]
        L.dt_tree_mask.restype = _i32
        L.dt_tree_mask.argtypes = [tp, _i32, _i32, _vp, _vp, _vp]
        L.dt_verify.restype = _i32
        L.dt_saba_budget.restype = _i32
        L.dt_saba_budget.argtypes = [ctypes.POINTER(SabaStruct), tp, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
        L.dt_verify_markov.restype = _i32
        L.dt_verify_markov.argtypes = [bp, tp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.dt_verify_rule.restype = _i32
        L.dt_verify_rule.argtypes = [tp, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
        L.dt_verify.argtypes = [tp, _i32, _i32, _i32, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp,
                                _vp]
        L.dt_select_dartree_noalloc.restype = _i32
        L.dt_select_dartree_noalloc.argtypes = [bp, tp, _vp]
        L.dt_test_wait_fault.restype = _i32
        L.dt_test_wait_fault.argtypes = [_i32, ctypes.c_int64]
        L.dt_status_str.restype = ctypes.c_char_p
        L.dt_status_str.argtypes = [_i32]
        L.dt_version.restype = _i32
        _LIB = L
    return _LIB


PROBE = {"stage1": 0x1, "walk": 0x2, "normaliser": 0x4}


def set_test_wait_fault(kernels=(), budget_cycles=2_000_000):
    """dt_test_wait_fault: make the named kernels' bounded waits run out once per
    staging step (a test of the timeout path); kernels=() turns it off."""
    mask = 0
    for k in kernels:
        mask |= PROBE[k]
    _check(lib().dt_test_wait_fault(mask, int(budget_cycles) if mask else 0), "dt_test_wait_fault")


class DtError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise DtError("%s: %s (%d)" % (what, lib().dt_status_str(rc).decode(), rc))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return DT_BF16
    if t.dtype == torch.float32:
        return DT_F32
    raise TypeError("logits must be bfloat16 or float32, got %s" % t.dtype)


def _need(t, dtype=None, name="tensor", numel=None):
    """A contiguous CUDA tensor (of dtype), holding at least numel elements: the
    C ABI takes bare pointers, so sizes are checked here, before any launch."""
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    _need_numel(t, numel, name)
    return t


def _need_numel(t, numel, name):
    if numel is not None and t.numel() < numel:
        raise ValueError("%s holds %d elements, the call reads or writes %d" % (name, t.numel(), numel))


def _need_batch(tree, batch):
    """The tree buffers (dt_tree carries no batch size) must hold `batch` requests."""
    if batch > tree.batch:
        raise ValueError("the tree buffers hold %d requests, the call covers %d" % (tree.batch, batch))


def _need_logits(t, p, name="draft_logits"):
    """[batch, L, V] drafter logits of Params p's dtype."""
    _need(t, name=name, numel=p.batch * p.L * p.V)
    if _dtype_code(t) != (DT_BF16 if p.dtype == "bf16" else DT_F32):
        raise TypeError("%s must be %s for dtype=%r, got %s" % (name, "bfloat16" if p.dtype == "bf16" else "float32",
                                                                p.dtype, t.dtype))
    if t.shape[-1] != p.V:
        raise ValueError("%s rows must hold V = %d logits, got %d" % (name, p.V, t.shape[-1]))


def _need_workspace(workspace):
    ws, n = (workspace if workspace is not None else (None, 0))
    if ws is not None:
        _need(ws, name="workspace")
        if ws.numel() * ws.element_size() < n:
            raise ValueError("workspace holds %d bytes, %d were declared" % (ws.numel() * ws.element_size(), n))
    return ws, n


@dataclasses.dataclass
class Params:
    """Build parameters; mirrors dt_build_params."""
    mode: str
    batch: int
    L: int
    V: int
    dtype: str = "bf16"
    K: int = 0
    B: int = 0
    W: int = 0
    beta: float = 0.0
    R: int = 0
    U: torch.Tensor = None
    Vt: torch.Tensor = None
    root_tok: torch.Tensor = None
    talon_k: int = 0
    mu: float = 0.0
    N: int = 0
    markov_norm: bool = False  # DARTree: full-vocabulary normalised correction
    tdes: "Tdes" = None        # heap mode: TDES edge scorer
    budget_policy: str = "topb"  # DARTree: "uniform" = DARTree (fixed), per-depth widths from B
    budgets: torch.Tensor = None  # DDTree / heap: [batch] int32 per-request budgets (dt_build_params.budget)

    @property
    def Kc(self):
        return min(self.N, self.V) if self.mode == "talon" else self.K

    @property
    def budget(self):
        return self.N if self.mode == "talon" else self.B

    def struct(self, for_launch=True):
        """The dt_build_params block.  for_launch: check the device tensors it points
        to (the host-only queries, workspace_size and stage1_plan, read no tensor)."""
        log_mu = 0.0
        if self.mode == "talon":
            log_mu = float(torch.tensor(math.log(self.mu), dtype=torch.float64).float())
        bp = BuildParams(DT_MODE[self.mode], self.batch, self.L, self.V,
                         DT_BF16 if self.dtype == "bf16" else DT_F32, self.K, self.B, self.W,
                         self.beta, self.R if self.U is not None else 0, _ptr(self.U), _ptr(self.Vt),
                         _ptr(self.root_tok), self.talon_k, log_mu, self.N, int(bool(self.markov_norm)))
        if for_launch:
            if self.U is not None:
                _need(self.U, torch.float32, "U", numel=self.V * self.R)
                _need(self.Vt, torch.float32, "Vt", numel=self.V * self.R)
            if self.root_tok is not None:
                _need(self.root_tok, torch.int32, "root_tok", numel=self.batch)
            if self.budgets is not None:
                _need(self.budgets, torch.int32, "budgets", numel=self.batch)
        if self.tdes is not None:
            if for_launch:
                H = int(self.tdes.w.shape[0])
                _need_numel(self.tdes.Ap, self.V * H, "Ap")
                _need_numel(self.tdes.Ac, self.V * H, "Ac")
                _need_numel(self.tdes.Dd, self.L * H, "Dd")
            bp._tdes = self.tdes.struct()  # kept alive with the parameter block
            bp.tdes = ctypes.pointer(bp._tdes)
        bp.budget_policy = BUDGET_POLICY[self.budget_policy]
        if self.budgets is not None:
            bp.budget = _ptr(self.budgets)
        return bp


@dataclasses.dataclass
class Tdes:
    """TDES edge scorer (dt_tdes): per-token first-layer rows Ap, Ac [V, H], depth rows
    Dd [L, H] (bias included), output weights w [H], bias b0, scale s; fp32 device tensors."""
    Ap: torch.Tensor
    Ac: torch.Tensor
    Dd: torch.Tensor
    w: torch.Tensor
    b0: float = 0.0
    s: float = 1.0

    def struct(self):
        for name in ("Ap", "Ac", "Dd", "w"):
            _need(getattr(self, name), torch.float32, name)
        return TdesStruct(int(self.w.shape[0]), _ptr(self.Ap), _ptr(self.Ac), _ptr(self.Dd), _ptr(self.w),
                          float(self.b0), float(self.s))


class TreeBuffers:
    """Device buffers of a batch of trees (dt_tree)."""

    def __init__(self, batch, L, Kc, max_nodes, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.batch, self.L, self.Kc, self.max_nodes = batch, L, Kc, max_nodes
        self.node_tok = torch.full((batch, max_nodes), -1, **i32)
        self.parent = torch.full((batch, max_nodes), -1, **i32)
        self.depth = torch.zeros((batch, max_nodes), **i32)
        self.rank = torch.full((batch, max_nodes), -1, **i32)
        self.score = torch.zeros((batch, max_nodes), **f32)
        self.n_nodes = torch.zeros((batch,), **i32)
        self.lse = torch.zeros((batch, L), **f32)
        self.cand_id = torch.zeros((batch, L, Kc), **i32)
        self.cand_lp = torch.zeros((batch, L, Kc), **f32)
        self.status = torch.zeros((batch,), **i32)

    def struct(self):
        return TreeStruct(self.max_nodes, self.Kc, self.L, *[
            _ptr(getattr(self, f)) for f in ("node_tok", "parent", "depth", "rank", "score", "n_nodes",
                                             "lse", "cand_id", "cand_lp", "status")])

    @classmethod
    def for_params(cls, p, max_nodes=None, device="cuda"):
        return cls(p.batch, p.L, p.Kc, max_nodes or p.budget + 1, device)


def workspace_size(p):
    ok = ctypes.c_int(0)
    n = lib().dt_workspace_size(ctypes.byref(p.struct(for_launch=False)), ctypes.byref(ok))
    if not ok.value:
        raise DtError("invalid parameters for dt_workspace_size")
    return int(n)


def make_workspace(p, device="cuda"):
    n = workspace_size(p)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device), n


def candidates(p, draft_logits, tree, stream=None):
    _need_logits(draft_logits, p)
    _need_batch(tree, p.batch)
    _check(lib().dt_candidates(ctypes.byref(p.struct()), _ptr(draft_logits), ctypes.byref(tree.struct()),
                               _stream(stream)), "dt_candidates")



def stage1_plan(p):
    """(kernel, cluster) that candidates() launches for Params p: kernel is
    "cluster" (each row over a cluster of `cluster` CTAs) or "rows" (a CTA per row)."""
    k, c = _i32(0), _i32(0)
    _check(lib().dt_stage1_plan(ctypes.byref(p.struct(for_launch=False)), ctypes.byref(k), ctypes.byref(c)),
           "dt_stage1_plan")
    return ({DT_STAGE1_CLUSTER: "cluster", DT_STAGE1_ROWS: "rows"}[k.value], c.value)

def stage1_ceiling(p, draft_logits, chunk_max, status=None, stream=None):
    """The read floor of the cluster stage-1 launch (dt_stage1_ceiling): every
    CTA's chunk maximum into chunk_max [batch * L, S] fp32, S from stage1_plan."""
    kind, S = stage1_plan(p)
    if kind != "cluster":
        raise DtError("dt_stage1_ceiling: the stage-1 plan for these parameters is one CTA per row")
    _need_logits(draft_logits, p)
    _need(chunk_max, torch.float32, "chunk_max", numel=p.batch * p.L * S)
    if status is not None:
        _need(status, torch.int32, "status", numel=1)
    _check(lib().dt_stage1_ceiling(ctypes.byref(p.struct()), _ptr(draft_logits), _ptr(chunk_max), _ptr(status),
                                   _stream(stream)), "dt_stage1_ceiling")


def markov_norm(p, draft_logits, tree, workspace, stream=None):
    """Full-vocabulary DARTree log-normalisers into the workspace (dt_markov_norm)."""
    _need_logits(draft_logits, p)
    _need_batch(tree, p.batch)
    ws, n = _need_workspace(workspace)
    _check(lib().dt_markov_norm(ctypes.byref(p.struct()), _ptr(draft_logits), ctypes.byref(tree.struct()), _ptr(ws),
                                n, _stream(stream)), "dt_markov_norm")


def znorm_view(p, workspace):
    """The [batch, L, K] fp32 log-normaliser table inside a DARTree workspace."""
    ws, _ = workspace
    off = (p.batch * p.L * p.K * p.K * 4 + 255) & ~255
    n = p.batch * p.L * p.K
    return ws[off:off + 4 * n].view(torch.float32).view(p.batch, p.L, p.K)


def select(p, tree, workspace=None, stream=None):
    _need_batch(tree, p.batch)
    ws, n = _need_workspace(workspace)
    _check(lib().dt_select(ctypes.byref(p.struct()), ctypes.byref(tree.struct()), _ptr(ws), n, _stream(stream)),
           "dt_select")


def select_dartree_noalloc(p, tree, stream=None):
    """DARTree selection with the library's own fixed table (no workspace);
    see dt_select_dartree_noalloc in include/dtree.h."""
    _need_batch(tree, p.batch)
    _check(lib().dt_select_dartree_noalloc(ctypes.byref(p.struct()), ctypes.byref(tree.struct()), _stream(stream)),
           "dt_select_dartree_noalloc")


def build_tree(p, draft_logits, tree, workspace=None, stream=None):
    """Stage 1 + selection.  workspace: (tensor, bytes) from make_workspace (DARTree)."""
    _need_logits(draft_logits, p)
    _need_batch(tree, p.batch)
    ws, n = _need_workspace(workspace)
    _check(lib().dt_build_tree(ctypes.byref(p.struct()), _ptr(draft_logits), ctypes.byref(tree.struct()),
                               _ptr(ws), n, _stream(stream)), "dt_build_tree")



def select_mask(p, tree, mask, pos, workspace=None, pos_offset=0, stream=None):
    """select + tree_mask with the mask written by the selection kernel (dt_select_mask)."""
    _need_batch(tree, p.batch)
    _need_mask(tree, p.batch, mask, pos)
    ws, n = _need_workspace(workspace)
    _check(lib().dt_select_mask(ctypes.byref(p.struct()), ctypes.byref(tree.struct()), _ptr(ws), n, int(pos_offset),
                                _ptr(mask), _ptr(pos), _stream(stream)), "dt_select_mask")


def build_tree_mask(p, draft_logits, tree, mask, pos, workspace=None, pos_offset=0, stream=None):
    """build_tree + tree_mask with the mask written by the selection kernel
    (dt_build_tree_mask); mask, pos from alloc_mask(tree)."""
    _need_logits(draft_logits, p)
    _need_batch(tree, p.batch)
    _need_mask(tree, p.batch, mask, pos)
    ws, n = _need_workspace(workspace)
    _check(lib().dt_build_tree_mask(ctypes.byref(p.struct()), _ptr(draft_logits), ctypes.byref(tree.struct()),
                                    _ptr(ws), n, int(pos_offset), _ptr(mask), _ptr(pos), _stream(stream)),
           "dt_build_tree_mask")

def tree_mask(tree, mask, pos, pos_offset=0, batch=None, stream=None):
    batch = batch or tree.batch
    _need_batch(tree, batch)
    _need_mask(tree, batch, mask, pos)
    _check(lib().dt_tree_mask(ctypes.byref(tree.struct()), batch, pos_offset, _ptr(mask), _ptr(pos),
                              _stream(stream)), "dt_tree_mask")


def _need_mask(tree, batch, mask, pos):
    words = (tree.max_nodes + 31) // 32
    _need(mask, torch.int32, "mask", numel=batch * tree.max_nodes * words)
    _need(pos, torch.int32, "pos", numel=batch * tree.max_nodes)


def _need_verify_io(tree, batch, V, draft, uniforms, target_lse, out, visited_lse):
    if draft is not None:
        _need(draft, name="draft", numel=batch * tree.L * V)
        if draft.shape[-1] != V:
            raise ValueError("draft rows must hold V = %d logits, got %d" % (V, draft.shape[-1]))
    if uniforms is not None:
        _need(uniforms, torch.float32, "uniforms", numel=batch * 2 * tree.max_nodes)
    if target_lse is not None:
        _need(target_lse, torch.float32, "target_lse", numel=batch * tree.max_nodes)
    acc_nodes, acc_len, next_tok = out
    _need(acc_nodes, torch.int32, "acc_nodes", numel=batch * (tree.L + 1))
    _need(acc_len, torch.int32, "acc_len", numel=batch)
    _need(next_tok, torch.int32, "next_tok", numel=batch)
    if visited_lse is not None:
        _need(visited_lse, torch.float32, "visited_lse", numel=batch * (tree.L + 1))


def alloc_mask(tree, device="cuda"):
    words = (tree.max_nodes + 31) // 32
    mask = torch.zeros((tree.batch, tree.max_nodes, words), dtype=torch.int32, device=device)
    pos = torch.zeros((tree.batch, tree.max_nodes), dtype=torch.int32, device=device)
    return mask, pos


def verify(tree, target, temperature=0.0, draft=None, uniforms=None, out=None, visited_lse=None, batch=None,
           target_lse=None, stream=None, rule=None):
    """Acceptance walk.  out = (acc_nodes [b, L+1], acc_len [b], next_tok [b]) int32 tensors;
    target_lse: optional [b, max_nodes] fp32 normalisers of the target rows (T=1);
    rule: None (greedy at temperature 0, "ratio" at 1) or one of VERIFY_RULES."""
    batch = batch or tree.batch
    _need_batch(tree, batch)
    V = target.shape[-1]
    _need(target, name="target", numel=batch * tree.max_nodes * V)
    if draft is not None and draft.dtype != target.dtype:
        # the walk reads both row sets with the target's element type
        raise TypeError("draft logits (%s) and target logits (%s) must share one dtype" % (draft.dtype, target.dtype))
    if out is None:
        out = alloc_verify_out(tree)
    acc_nodes, acc_len, next_tok = out
    _need_verify_io(tree, batch, V, draft, uniforms, target_lse, out, visited_lse)
    if rule is not None:
        _check(lib().dt_verify_rule(ctypes.byref(tree.struct()), batch, V, _dtype_code(target), _ptr(target),
                                    _ptr(target_lse), _ptr(draft), VERIFY_RULES[rule], _ptr(uniforms),
                                    _ptr(acc_nodes), _ptr(acc_len), _ptr(next_tok), _ptr(visited_lse),
                                    _stream(stream)), "dt_verify_rule")
        return out
    _check(lib().dt_verify(ctypes.byref(tree.struct()), batch, V, _dtype_code(target), _ptr(target),
                           _ptr(target_lse), _ptr(draft), float(temperature), _ptr(uniforms), _ptr(acc_nodes),
                           _ptr(acc_len), _ptr(next_tok), _ptr(visited_lse), _stream(stream)), "dt_verify")
    return out


def verify_markov(p, tree, target, draft, znorm, uniforms, out=None, visited_lse=None, target_lse=None,
                  stream=None):
    """T=1 walk against the normalised DARTree proposal (dt_verify_markov); znorm [b, L, K] fp32,
    e.g. znorm_view(p, workspace) after markov_norm."""
    _need_batch(tree, p.batch)
    _need(target, name="target", numel=p.batch * tree.max_nodes * p.V)
    _need_logits(draft, p, "draft")
    if _dtype_code(target) != _dtype_code(draft):
        # the walk reads the target rows with the parameter block's element type
        raise TypeError("target logits must be %s for dtype=%r, got %s" % (draft.dtype, p.dtype, target.dtype))
    _need(znorm, torch.float32, "znorm", numel=p.batch * p.L * p.K)
    if out is None:
        out = alloc_verify_out(tree)
    acc_nodes, acc_len, next_tok = out
    _need_verify_io(tree, p.batch, p.V, None, uniforms, target_lse, out, visited_lse)
    if uniforms is None:
        raise ValueError("verify_markov needs uniforms")
    _check(lib().dt_verify_markov(ctypes.byref(p.struct()), ctypes.byref(tree.struct()), _ptr(target),
                                  _ptr(target_lse), _ptr(draft), _ptr(znorm), _ptr(uniforms), _ptr(acc_nodes),
                                  _ptr(acc_len), _ptr(next_tok), _ptr(visited_lse), _stream(stream)),
           "dt_verify_markov")
    return out


def alloc_verify_out(tree, device="cuda"):
    return (torch.full((tree.batch, tree.L + 1), -1, dtype=torch.int32, device=device),
            torch.zeros((tree.batch,), dtype=torch.int32, device=device),
            torch.zeros((tree.batch,), dtype=torch.int32, device=device))


class SabaState:
    """Device SABA history for a batch: ring [batch, window] and count [batch] (int32, zeroed)."""

    def __init__(self, batch, window, device="cuda"):
        self.window = window
        self.ring = torch.zeros((batch, window), dtype=torch.int32, device=device)
        self.count = torch.zeros((batch,), dtype=torch.int32, device=device)


def saba_budget(tree, st, c_verify, c_fixed, B_min, B_max, budget, state, hidden=None, prev_acc_len=None,
                batch=None, stream=None):
    """dt_saba_budget: per-request budgets [batch] int32 and state [batch, 4] fp32 (conf, degen, hist, a);
    hidden: optional [batch, L, Hd] fp32 drafter hidden states; prev_acc_len: last round's acc_len."""
    batch = batch or tree.batch
    _need_batch(tree, batch)
    _need(budget, torch.int32, "budget", numel=batch)
    _need(state, torch.float32, "state", numel=batch * 4)
    _need(st.ring, torch.int32, "ring", numel=batch * st.window)
    _need(st.count, torch.int32, "count", numel=batch)
    Hd = 0
    if hidden is not None:
        Hd = int(hidden.shape[-1])
        _need(hidden, torch.float32, "hidden", numel=batch * tree.L * Hd)
    if prev_acc_len is not None:
        _need(prev_acc_len, torch.int32, "prev_acc_len", numel=batch)
    q = SabaStruct(st.window, float(c_verify), float(c_fixed), int(B_min), int(B_max))
    _check(lib().dt_saba_budget(ctypes.byref(q), ctypes.byref(tree.struct()), batch, _ptr(hidden), Hd,
                                _ptr(prev_acc_len), _ptr(st.ring), _ptr(st.count), _ptr(state), _ptr(budget),
                                _stream(stream)), "dt_saba_budget")
