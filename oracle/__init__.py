"""CPU oracle for draft-tree build and tree verification -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is a plain, slow restatement of the
method in C (``dt_oracle.c``) with numpy-level wrappers; it shares no code with
the CUDA path.  See ``dt_oracle.c`` for the passage each function follows and
for what pins it.
"""
import ctypes
import dataclasses
import os

import numpy as np

from . import build as _build
from .endtoend import path_scores, selection_check  # noqa: F401  (end-to-end selection check)

_LIB = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i64p = ctypes.POINTER(ctypes.c_int64)


def lib():
    global _LIB
    if _LIB is None:
        # DT_ORACLE_LIB: another build of the oracle source (the mutation tests
        # load deliberately broken copies this way, one per process)
        path = os.environ.get("DT_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        L.or_exp_canon.restype = ctypes.c_float
        L.or_exp_canon.argtypes = [ctypes.c_float]
        L.or_exp_canon_vec.argtypes = [_f32p, ctypes.c_int64, _f32p]
        L.or_candidates.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                    _f64p, _f32p, _i32p, _f32p]
        L.or_ddtree.argtypes = [_f32p, _i32p] + [ctypes.c_int] * 5 + [_i32p] * 4 + [_f32p, _i32p]
        L.or_dartree.argtypes = ([_f32p, _i32p, ctypes.c_int, ctypes.c_int, _f32p, _f32p,
                                  ctypes.c_int, ctypes.c_int, _f32p, ctypes.c_int, _i32p, ctypes.c_float,
                                  ctypes.c_int, ctypes.c_int] + [_i32p] * 4 +
                                 [_f32p, _i32p, _i32p, _i32p])
        L.or_uniform_widths.argtypes = [ctypes.c_int, ctypes.c_int, _i32p]
        L.or_saba.argtypes = [_f32p, ctypes.c_int, _f32p, ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                              ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int, _f32p, _i32p]
        L.or_markov_norm.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _f32p, _f32p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p]
        L.or_markov_table.argtypes = [_i32p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, ctypes.c_int,
                                      ctypes.c_int, _f32p]
        L.or_tdes_table.argtypes = [_i32p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, _f32p, _f32p, ctypes.c_int,
                                    ctypes.c_float, ctypes.c_float, ctypes.c_int, _f32p]
        L.or_heap_select.argtypes = ([_f32p, _i32p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, ctypes.c_int,
                                      ctypes.c_int] + [_i32p] * 4 + [_f32p, _i32p])
        L.or_talon.argtypes = ([_f32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_float, ctypes.c_int, ctypes.c_int] + [_i32p] * 4 +
                               [_f32p, _i32p])
        L.or_tree_mask.argtypes = [_i32p, _i32p] + [ctypes.c_int] * 4 + [_u32p, _i32p]
        L.or_verify_greedy.argtypes = ([_i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                        _f32p, ctypes.c_int, _i32p, _i32p, _i32p])
        L.or_verify_t1.argtypes = ([_i32p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, _f32p, _f32p, _f32p, ctypes.c_int, _f32p,
                                    _f32p, _i32p, _i32p, _i32p, _f32p])
        L.or_verify_iter_residual.argtypes = L.or_verify_t1.argtypes
        L.or_verify_t1_markov.argtypes = ([_i32p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _f32p, _f32p, _f32p, ctypes.c_int, _f32p, _f32p, ctypes.c_int,
                                           ctypes.c_int, _f32p, ctypes.c_int, _f32p, _f32p, _i32p, _i32p, _i32p])
        L.or_verify_target_match.argtypes = ([_i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              _f32p, ctypes.c_int, _f32p, _f32p, _i32p, _i32p, _i32p, _f32p])
        L.or_spec_scalar.argtypes = [_f64p, _f64p, ctypes.c_int, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_double, _f64p, _f64p, _i32p]
        L.or_spec_scalar_trials.argtypes = [_f64p, _f64p, ctypes.c_int, _f64p,
                                            ctypes.c_int64, _i64p]
        _LIB = L
    return _LIB


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed with code %d" % (what, rc))


@dataclasses.dataclass
class Tree:
    """Flattened draft tree; node 0 is the root (token -1, parent -1)."""
    tok: np.ndarray
    parent: np.ndarray
    depth: np.ndarray
    rank: np.ndarray
    score: np.ndarray
    n: int

    def trimmed(self):
        n = self.n
        return Tree(self.tok[:n].copy(), self.parent[:n].copy(), self.depth[:n].copy(),
                    self.rank[:n].copy(), self.score[:n].copy(), n)


def _new_tree(Mmax):
    return Tree(np.full(Mmax, -1, np.int32), np.full(Mmax, -1, np.int32),
                np.zeros(Mmax, np.int32), np.full(Mmax, -1, np.int32),
                np.zeros(Mmax, np.float32), 0)


def _tree_args(t):
    return [_p(t.tok, ctypes.c_int32), _p(t.parent, ctypes.c_int32),
            _p(t.depth, ctypes.c_int32), _p(t.rank, ctypes.c_int32),
            _p(t.score, ctypes.c_float)]


def exp_canon(x):
    x = _f32(x)
    y = np.empty_like(x)
    lib().or_exp_canon_vec(_p(x, ctypes.c_float), x.size, _p(y, ctypes.c_float))
    return y


def candidates(x, Kc):
    """Per-row log-normaliser and Top-Kc list of a [rows, V] logit array.

    Returns (lse64, lse32, ids [rows, Kc], lps [rows, Kc])."""
    x = _f32(x)
    rows, V = x.reshape(-1, x.shape[-1]).shape
    lse64 = np.empty(rows, np.float64)
    lse32 = np.empty(rows, np.float32)
    ids = np.empty((rows, Kc), np.int32)
    lps = np.empty((rows, Kc), np.float32)
    _check(lib().or_candidates(_p(x, ctypes.c_float), rows, V, Kc, _p(lse64, ctypes.c_double),
                               _p(lse32, ctypes.c_float), _p(ids, ctypes.c_int32),
                               _p(lps, ctypes.c_float)), "candidates")
    return lse64, lse32, ids, lps


def ddtree(cand_lp, cand_id, B, Mmax=None, rule=0):
    """DDTree Top-B by the literal heap; cand_* are [L, K] rank-ordered lists."""
    lp = _f32(cand_lp)
    ids = _i32(cand_id)
    L, K = lp.shape
    Mmax = Mmax or B + 1
    t = _new_tree(Mmax)
    n = np.zeros(1, np.int32)
    _check(lib().or_ddtree(_p(lp, ctypes.c_float), _p(ids, ctypes.c_int32), L, K, B, rule,
                           Mmax, *_tree_args(t), _p(n, ctypes.c_int32)), "ddtree")
    t.n = int(n[0])
    return t


def uniform_widths(B, L):
    """DARTree (fixed): per-depth widths spreading B over L depths."""
    w = np.zeros(L, np.int32)
    _check(lib().or_uniform_widths(B, L, _p(w, ctypes.c_int32)), "uniform_widths")
    return w


class SabaState:
    """One request's SABA history: a ring of the last w accepted lengths and a count."""

    def __init__(self, w):
        self.w = w
        self.ring = np.zeros(w, np.int32)
        self.count = np.zeros(1, np.int32)


def saba(top_lp, hidden, st, prev_len, c_verify, c_fixed, B_min, B_max):
    """SABA budget for one request: top_lp [D] (lp of each position's top candidate),
    hidden [D, Hd] or None, st a SabaState (updated), prev_len the last round's
    accepted length or -1.  Returns (budget, state [conf, degen, hist, a])."""
    lp = _f32(top_lp)
    D = lp.shape[0]
    hp, Hd = None, 0
    if hidden is not None:
        hidden = _f32(hidden)
        hp, Hd = _p(hidden, ctypes.c_float), hidden.shape[1]
    state = np.zeros(4, np.float32)
    b = np.zeros(1, np.int32)
    _check(lib().or_saba(_p(lp, ctypes.c_float), D, hp, Hd, _p(st.ring, ctypes.c_int32),
                         _p(st.count, ctypes.c_int32), st.w, int(prev_len), ctypes.c_float(c_verify),
                         ctypes.c_float(c_fixed), B_min, B_max, _p(state, ctypes.c_float), _p(b, ctypes.c_int32)),
           "saba")
    return int(b[0]), state


def dartree(cand_lp, cand_id, U, Vt, root_tok, W, beta, B, Mmax=None, znorm=None, widths=None):
    """DARTree supertree + deferred pruning.  Returns (tree, info, topb) with
    info = dict(topb_equals_bestfirst, violations, supertree_size).  znorm
    ([L, K] fp32 log-normalisers from markov_norm) selects the full-vocabulary
    normalised correction."""
    lp = _f32(cand_lp)
    ids = _i32(cand_id)
    L, K = lp.shape
    if U is None:
        Up = Vp = None
        R = 0
    else:
        U = _f32(U)
        Vt = _f32(Vt)
        R = U.shape[1]
        Up, Vp = _p(U, ctypes.c_float), _p(Vt, ctypes.c_float)
    zp = None
    if znorm is not None:
        znorm = _f32(znorm).reshape(L, K)
        zp = _p(znorm, ctypes.c_float)
    Mmax = Mmax or B + 1
    t = _new_tree(Mmax)
    n = np.zeros(1, np.int32)
    info = np.zeros(3, np.int32)
    topb = np.full(Mmax, -1, np.int32)
    wp = None
    if widths is not None:
        widths = _i32(widths)
        wp = _p(widths, ctypes.c_int32)
    _check(lib().or_dartree(_p(lp, ctypes.c_float), _p(ids, ctypes.c_int32), L, K, Up, Vp, R,
                            int(root_tok), zp, W, wp, ctypes.c_float(beta), B, Mmax, *_tree_args(t),
                            _p(n, ctypes.c_int32), _p(info, ctypes.c_int32),
                            _p(topb, ctypes.c_int32)), "dartree")
    t.n = int(n[0])
    return t, dict(topb_equals_bestfirst=bool(info[0]), violations=int(info[1]),
                   supertree_size=int(info[2])), topb


def markov_table(cand_id, U, Vt, root_tok):
    """[L, K, K] Markov edge terms <U[parent], Vt[child]> on the candidate lattice
    (row 0 of position 0: the root token; zeros when root_tok < 0)."""
    ids = _i32(cand_id)
    L, K = ids.shape
    U, Vt = _f32(U), _f32(Vt)
    E = np.empty((L, K, K), np.float32)
    _check(lib().or_markov_table(_p(ids, ctypes.c_int32), L, K, _p(U, ctypes.c_float), _p(Vt, ctypes.c_float),
                                 U.shape[1], int(root_tok), _p(E, ctypes.c_float)), "markov_table")
    return E


def tdes_table(cand_id, Ap, Ac, Dd, w, b0, s, root_tok):
    """[L, K, K] TDES edge terms s * f(parent, child, depth) on the candidate lattice.
    Ap, Ac: [V, H] per-token first-layer rows; Dd: [L, H] depth rows (bias included); w: [H]."""
    ids = _i32(cand_id)
    L, K = ids.shape
    Ap, Ac, Dd, w = _f32(Ap), _f32(Ac), _f32(Dd), _f32(w)
    H = w.shape[0]
    E = np.empty((L, K, K), np.float32)
    _check(lib().or_tdes_table(_p(ids, ctypes.c_int32), L, K, _p(Ap, ctypes.c_float), _p(Ac, ctypes.c_float),
                               _p(Dd, ctypes.c_float), _p(w, ctypes.c_float), H, ctypes.c_float(b0),
                               ctypes.c_float(s), int(root_tok), _p(E, ctypes.c_float)), "tdes_table")
    return E


def heap_select(cand_lp, cand_id, B, E=None, znorm=None, Mmax=None):
    """Best-first heap with parent-conditioned edge scores lp + E (- znorm);
    E: [L, K, K] from markov_table / tdes_table, or None (DDTree)."""
    lp = _f32(cand_lp)
    ids = _i32(cand_id)
    L, K = lp.shape
    Ep = zp = None
    if E is not None:
        E = _f32(E).reshape(L, K, K)
        Ep = _p(E, ctypes.c_float)
    if znorm is not None:
        znorm = _f32(znorm).reshape(L, K)
        zp = _p(znorm, ctypes.c_float)
    Mmax = Mmax or B + 1
    t = _new_tree(Mmax)
    n = np.zeros(1, np.int32)
    _check(lib().or_heap_select(_p(lp, ctypes.c_float), _p(ids, ctypes.c_int32), L, K, Ep, zp, B, Mmax,
                                *_tree_args(t), _p(n, ctypes.c_int32)), "heap_select")
    t.n = int(n[0])
    return t


def markov_norm(x, cand_id, U, Vt, root_tok, only_row=-1, out=None):
    """[L, K] fp32 log-normalisers log Z of the full-vocabulary corrected
    distribution (double inside) for raw logits x [L, V] (fp32 values) and the
    candidate ids [L, K]; only_row >= 0 computes that flat row alone."""
    x = _f32(x)
    ids = _i32(cand_id)
    L, V = x.shape
    K = ids.shape[1]
    U = _f32(U)
    Vt = _f32(Vt)
    z = np.zeros((L, K), np.float32) if out is None else out
    _check(lib().or_markov_norm(_p(x, ctypes.c_float), L, V, _p(ids, ctypes.c_int32), K, _p(U, ctypes.c_float),
                                _p(Vt, ctypes.c_float), U.shape[1], int(root_tok), int(only_row),
                                _p(z, ctypes.c_float)), "markov_norm")
    return z


def talon(cand_lp, cand_id, talon_k, log_mu, N, Mmax=None):
    lp = _f32(cand_lp)
    ids = _i32(cand_id)
    L, Kc = lp.shape
    Mmax = Mmax or N + 1
    t = _new_tree(Mmax)
    n = np.zeros(1, np.int32)
    _check(lib().or_talon(_p(lp, ctypes.c_float), _p(ids, ctypes.c_int32), L, Kc, talon_k,
                          ctypes.c_float(log_mu), N, Mmax, *_tree_args(t),
                          _p(n, ctypes.c_int32)), "talon")
    t.n = int(n[0])
    return t


def tree_mask(tree, Mmax, L, pos_offset=0):
    """Returns (status, mask [Mmax, ceil(Mmax/32)] uint32, pos [Mmax])."""
    words = (Mmax + 31) // 32
    mask = np.zeros((Mmax, words), np.uint32)
    pos = np.zeros(Mmax, np.int32)
    par = _i32(tree.parent)
    dep = _i32(tree.depth)
    rc = lib().or_tree_mask(_p(par, ctypes.c_int32), _p(dep, ctypes.c_int32), tree.n, Mmax, L,
                            pos_offset, _p(mask, ctypes.c_uint32), _p(pos, ctypes.c_int32))
    return rc, mask, pos


def verify_greedy(tree, target, L):
    """target: [>= tree.n, V] rows indexed by node.  Returns (acc_nodes, acc_len, next_tok)."""
    target = _f32(target)
    V = target.shape[-1]
    acc = np.empty(L + 1, np.int32)
    alen = np.zeros(1, np.int32)
    nxt = np.zeros(1, np.int32)
    tok, par, dep = _i32(tree.tok), _i32(tree.parent), _i32(tree.depth)
    rc = lib().or_verify_greedy(_p(tok, ctypes.c_int32), _p(par, ctypes.c_int32),
                                _p(dep, ctypes.c_int32), tree.n, L, _p(target, ctypes.c_float),
                                V, _p(acc, ctypes.c_int32), _p(alen, ctypes.c_int32),
                                _p(nxt, ctypes.c_int32))
    _check(rc, "verify_greedy")
    return acc, int(alen[0]), int(nxt[0])


def verify_t1(tree, target, draft, draft_lse, uniforms, L, Mmax, lse_in=None, rule="ratio"):
    """uniforms: [2, Mmax] (row 0: per-child acceptance, row 1: per-node draw);
    lse_in: optional per-node target normalisers [Mmax];
    rule: "ratio" (every child against p), "iter_residual" (one residual per
    rejected sibling) or "target_match" (draw from the target, match a child;
    draft and draft_lse unused).
    Returns (acc_nodes, acc_len, next_tok, lse_used per step [L+1])."""
    if rule == "target_match":
        return verify_target_match(tree, target, uniforms, L, Mmax, lse_in)
    target = _f32(target)
    draft = _f32(draft)
    draft_lse = _f32(draft_lse)
    u = _f32(uniforms)
    assert u.shape == (2, Mmax)
    V = target.shape[-1]
    acc = np.empty(L + 1, np.int32)
    alen = np.zeros(1, np.int32)
    nxt = np.zeros(1, np.int32)
    lse_out = np.zeros(L + 1, np.float32)
    tok, par, dep, rnk = _i32(tree.tok), _i32(tree.parent), _i32(tree.depth), _i32(tree.rank)
    lin = None
    if lse_in is not None:
        lse_in = _f32(lse_in)
        lin = _p(lse_in, ctypes.c_float)
    fn = {"ratio": lib().or_verify_t1, "iter_residual": lib().or_verify_iter_residual}[rule]
    rc = fn(_p(tok, ctypes.c_int32), _p(par, ctypes.c_int32),
                            _p(dep, ctypes.c_int32), _p(rnk, ctypes.c_int32), tree.n, L, Mmax,
                            _p(target, ctypes.c_float), _p(draft, ctypes.c_float),
                            _p(draft_lse, ctypes.c_float), V, _p(u, ctypes.c_float), lin,
                            _p(acc, ctypes.c_int32), _p(alen, ctypes.c_int32),
                            _p(nxt, ctypes.c_int32), _p(lse_out, ctypes.c_float))
    _check(rc, "verify_t1 " + rule)
    return acc, int(alen[0]), int(nxt[0]), lse_out


def verify_t1_markov(tree, target, draft, draft_lse, U, Vt, root_tok, znorm, uniforms, L, Mmax, lse_in=None):
    """T=1 walk against the normalised DARTree proposal q~(. | parent token);
    znorm: [L, K] log-normalisers (markov_norm).  Returns (acc_nodes, acc_len, next_tok)."""
    target, draft, draft_lse = _f32(target), _f32(draft), _f32(draft_lse)
    U, Vt, z, u = _f32(U), _f32(Vt), _f32(znorm), _f32(uniforms)
    assert u.shape == (2, Mmax)
    V = target.shape[-1]
    acc = np.empty(L + 1, np.int32)
    alen = np.zeros(1, np.int32)
    nxt = np.zeros(1, np.int32)
    tok, par, dep, rnk = _i32(tree.tok), _i32(tree.parent), _i32(tree.depth), _i32(tree.rank)
    lin = None
    if lse_in is not None:
        lse_in = _f32(lse_in)
        lin = _p(lse_in, ctypes.c_float)
    rc = lib().or_verify_t1_markov(_p(tok, ctypes.c_int32), _p(par, ctypes.c_int32), _p(dep, ctypes.c_int32),
                                   _p(rnk, ctypes.c_int32), tree.n, L, Mmax, _p(target, ctypes.c_float),
                                   _p(draft, ctypes.c_float), _p(draft_lse, ctypes.c_float), V,
                                   _p(U, ctypes.c_float), _p(Vt, ctypes.c_float), U.shape[1], int(root_tok),
                                   _p(z, ctypes.c_float), z.shape[-1], _p(u, ctypes.c_float), lin,
                                   _p(acc, ctypes.c_int32), _p(alen, ctypes.c_int32), _p(nxt, ctypes.c_int32))
    _check(rc, "verify_t1_markov")
    return acc, int(alen[0]), int(nxt[0])


def verify_target_match(tree, target, uniforms, L, Mmax, lse_in=None):
    """Exact target-sample matching; uniforms [2, Mmax] (row 1 used).
    Returns (acc_nodes, acc_len, next_tok, lse_used per step [L+1])."""
    target = _f32(target)
    u = _f32(uniforms)
    assert u.shape == (2, Mmax)
    V = target.shape[-1]
    acc = np.empty(L + 1, np.int32)
    alen = np.zeros(1, np.int32)
    nxt = np.zeros(1, np.int32)
    lse_out = np.zeros(L + 1, np.float32)
    tok, par, dep = _i32(tree.tok), _i32(tree.parent), _i32(tree.depth)
    lin = None
    if lse_in is not None:
        lse_in = _f32(lse_in)
        lin = _p(lse_in, ctypes.c_float)
    rc = lib().or_verify_target_match(_p(tok, ctypes.c_int32), _p(par, ctypes.c_int32), _p(dep, ctypes.c_int32),
                                      tree.n, L, Mmax, _p(target, ctypes.c_float), V, _p(u, ctypes.c_float), lin,
                                      _p(acc, ctypes.c_int32), _p(alen, ctypes.c_int32), _p(nxt, ctypes.c_int32),
                                      _p(lse_out, ctypes.c_float))
    _check(rc, "verify_target_match")
    return acc, int(alen[0]), int(nxt[0]), lse_out


def spec_scalar(p, q, u_draw, u_acc, u_res):
    """Single-position rule in double.  Returns (emitted, drafted, accept_prob, residual)."""
    p = np.ascontiguousarray(p, np.float64)
    q = np.ascontiguousarray(q, np.float64)
    n = p.size
    a = np.empty(n)
    r = np.empty(n)
    d = np.zeros(1, np.int32)
    y = lib().or_spec_scalar(_p(p, ctypes.c_double), _p(q, ctypes.c_double), n, u_draw, u_acc,
                             u_res, _p(a, ctypes.c_double), _p(r, ctypes.c_double),
                             _p(d, ctypes.c_int32))
    return int(y), int(d[0]), a, r


def spec_scalar_trials(p, q, uniforms):
    p = np.ascontiguousarray(p, np.float64)
    q = np.ascontiguousarray(q, np.float64)
    u = np.ascontiguousarray(uniforms, np.float64).reshape(-1)
    trials = u.size // 3
    counts = np.zeros(p.size, np.int64)
    _check(lib().or_spec_scalar_trials(_p(p, ctypes.c_double), _p(q, ctypes.c_double), p.size,
                                       _p(u, ctypes.c_double), trials,
                                       _p(counts, ctypes.c_int64)), "spec_scalar_trials")
    return counts
