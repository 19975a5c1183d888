"""The oracle's pins catch plausible mistakes.

Each mutant below is the oracle's C source with one deliberate slip of the kind
a restatement of the pages could contain -- a dropped term, a flipped sign or
comparison, a transposed operand, an index off by one -- in each part of the
path (stage 1, the three selections, the budget policies, the edge tables, the
mask, the walks).  Every mutant is compiled beside the real oracle with the
same flags and loaded, in a child process, in its place (DT_ORACLE_LIB); the
pin tests named for it must then fail.  A control build of the unmodified
source must pass the same tests through the same harness, so that a broken
harness cannot pass for caught mutants.

The mistakes are planted only in temporary copies of the oracle on the CPU.
"""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

from oracle import build as oracle_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = "tests/test_oracle_pins.py"
BUDGETS = "tests/test_oracle_budgets.py"
NORM = "tests/test_oracle_markov_norm.py"
HEAP = "tests/test_oracle_heap_tdes.py"
VARIANTS = "tests/test_oracle_verify_variants.py"

# (name, exact source text (must occur once), replacement, pin files that must fail)
MUTANTS = [
    # stage 1: exponential, log-normaliser, rank order
    ("exp_drops_ln2_tail", "r = fmaf(-kf, ln2_lo, r);", "(void)ln2_lo;", [PINS]),
    ("exp_wrong_taylor_coefficient", "p = fmaf(p, r, 0.5f);", "p = fmaf(p, r, 0.25f);", [PINS]),
    ("lse_forgets_the_max", "double l = (m == -INFINITY) ? m : m + log(s);",
     "double l = (m == -INFINITY) ? m : log(s);", [PINS]),
    ("topk_ties_by_larger_id", "return (a->id < b->id) ? -1 : (a->id > b->id);",
     "return (a->id > b->id) ? -1 : (a->id < b->id);", [PINS]),
    ("lp_adds_the_normaliser", "float lp = buf[k].v - l32;", "float lp = buf[k].v + l32;", [PINS]),
    # node order and DDTree
    ("extension_before_prefix", "    return da < db;\n}", "    return da > db;\n}", [PINS]),
    ("score_subtracts_lp", "for (int i = 0; i < d; ++i) s = s + lp[i * K + r[i]];",
     "for (int i = 0; i < d; ++i) s = s - lp[i * K + r[i]];", [PINS]),
    ("ddtree_skips_a_sibling", "sib.r[sib.d - 1] += 1;", "sib.r[sib.d - 1] += 2;", [PINS]),
    ("ddtree_depth_cap_off_by_one", "int push_child = (x.d < L) &&", "int push_child = (x.d <= L) &&", [PINS]),
    # DARTree
    ("dartree_beta_sign", "x->s = (S[p].s + t) + beta;", "x->s = (S[p].s + t) - beta;", [PINS, NORM]),
    ("dartree_markov_transposed", "t = l + or_markov(U, Vt, R, ptok, c);",
     "t = l + or_markov(U, Vt, R, c, ptok);", [PINS, NORM]),
    ("dartree_keeps_one_too_many", "int keep = nk < Wd ? nk : Wd;", "int keep = nk < Wd + 1 ? nk : Wd + 1;",
     [PINS, BUDGETS]),
    ("dartree_norm_sign", "if (znorm != NULL) t = t - znorm[", "if (znorm != NULL) t = t + znorm[", [NORM, HEAP]),
    # budget policies
    ("widths_remainder_to_the_deepest", "widths[d] = B / L + (d < B % L ? 1 : 0);",
     "widths[d] = B / L + (d >= L - B % L ? 1 : 0);", [BUDGETS]),
    ("saba_largest_budget_on_ties", "if (u > bu) { bu = u; best = B; }", "if (u >= bu) { bu = u; best = B; }",
     [BUDGETS]),
    ("saba_growth_sign", "degen = rs / (D - 1) + (rl - r0);", "degen = rs / (D - 1) + (r0 - rl);", [BUDGETS]),
    ("saba_gain_exponent", "float u = (a * sqrtf((float)B))", "float u = (a * (float)B)", [BUDGETS]),
    # edge tables and the heap
    ("norm_drops_the_log_softmax", "a[v] = ((double)xd[v] - lse) + m;", "a[v] = (double)xd[v] + m;", [NORM]),
    ("markov_table_transposed", "= or_markov(U, Vt, R, ptok, id[d * K + j]);",
     "= or_markov(U, Vt, R, id[d * K + j], ptok);", [HEAP]),
    ("tdes_without_relu", "float r = a > 0.0f ? a : 0.0f;", "float r = a;", [HEAP]),
    ("tdes_drops_output_bias", "E[((int64_t)d * K + i) * K + j] = s * (acc + b0);",
     "E[((int64_t)d * K + i) * K + j] = s * acc;", [HEAP]),
    ("heap_norm_sign", "if (or_hs_z) t = t - or_hs_z[(d - 1) * K + i];",
     "if (or_hs_z) t = t + or_hs_z[(d - 1) * K + i];", [HEAP]),
    ("heap_sibling_under_wrong_row",
     "sib.s = score[p] + or_hs_edge(x.d, crank[p], ord[(size_t)p * K + jpos + 1]);",
     "sib.s = score[p] + or_hs_edge(x.d, c, ord[(size_t)p * K + jpos + 1]);", [HEAP]),
    # TALON
    ("talon_gate_sign", "float thr = m_d + log_mu;", "float thr = m_d - log_mu;", [PINS]),
    ("talon_gate_strict", "if (pool[i].s >= thr) pool[npass++] = pool[i];",
     "if (pool[i].s > thr) pool[npass++] = pool[i];", [PINS]),
    ("talon_root_layer_one_more", "int k1 = talon_k;", "int k1 = talon_k + 1;", [PINS]),
    # mask and positions
    ("mask_without_self", "for (int a = n; a != -1; a = parent[a])",
     "for (int a = parent[n]; a != -1; a = parent[a])", [PINS]),
    ("positions_ignore_offset", "pos[n] = depth[n] + pos_offset;", "pos[n] = depth[n];", [PINS]),
    # walks
    ("greedy_ties_to_larger_id", "if (row[v] > row[a]) a = v;", "if (row[v] >= row[a]) a = v;", [PINS]),
    ("t1_ratio_inverted", "float ratio = or_exp_canon(lpt - lpq);", "float ratio = or_exp_canon(lpq - lpt);",
     [PINS]),
    ("t1_residual_reversed", "(drow[v] - lsed));\n                w[v] = P > Q ? P - Q : 0;",
     "(drow[v] - lsed));\n                w[v] = Q > P ? Q - P : 0;", [PINS]),
    ("draw_prefix_off_by_one", "if (acc > target) return v;", "if (acc >= target) return v;", [PINS, VARIANTS]),
    ("iter_residual_unscaled", "return P > s ? P - s : 0;", "return P > Q ? P - Q : 0;", [VARIANTS]),
    ("markov_walk_norm_sign", "or_markov(U, Vt, R, ptok, tok[c]); lpq = lpq - z; }",
     "or_markov(U, Vt, R, ptok, tok[c]); lpq = lpq + z; }", [VARIANTS]),
    ("markov_residual_drops_the_term", "lpq = lpq + or_markov(U, Vt, R, ptok, v); lpq = lpq - z; }",
     "lpq = lpq - z; }", [VARIANTS]),
    ("target_match_wrong_uniform", "y = or_draw(w, V, S, u[Mmax + n]);", "y = or_draw(w, V, S, u[n]);", [VARIANTS]),
    ("scalar_residual_not_clipped", "residual[i] = z > 0.0 ? z : 0.0;", "residual[i] = z;", [PINS]),
    ("t1_drafter_row_off_by_one", "int pos = depth[c] - 1;", "int pos = depth[c];", [PINS]),
    ("t1_accept_wrong_uniform_row", "if (u[c] < ratio) acc = c;", "if (u[Mmax + c] < ratio) acc = c;", [PINS]),
    ("iter_accept_scale_halved", "unsigned __int128 rhs = (unsigned __int128)W << 56;",
     "unsigned __int128 rhs = (unsigned __int128)W << 55;", [VARIANTS]),
    ("t1_markov_every_parent_takes_rank0_norm",
     "if (ptok >= 0 && pos < L) z = znorm[pos * K + (n == 0 ? 0 : rank[n])];",
     "if (ptok >= 0 && pos < L) z = znorm[pos * K];", [VARIANTS]),
    # more of stage 1, the selections and the tables
    ("exp_underflows_early", "if (x < -86.0f) return 0.0f;", "if (x < -80.0f) return 0.0f;", [PINS]),
    ("markov_dot_drops_last_term", "for (int k = 0; k < R; ++k)\n        acc = fmaf(",
     "for (int k = 0; k < R - 1; ++k)\n        acc = fmaf(", [PINS, HEAP, NORM, VARIANTS]),
    ("dartree_depth1_skips_root_term", "if (U != NULL && ptok >= 0) {", "if (U != NULL && ptok >= 0 && d > 1) {",
     [PINS, NORM]),
    ("ddtree_budget_plus_one",
     "while (rc == OR_OK && n < B && h.n > 0) {\n        or_node x = or_heap_pop(&h);\n        /* the parent",
     "while (rc == OR_OK && n <= B && h.n > 0) {\n        or_node x = or_heap_pop(&h);\n        /* the parent",
     [PINS]),
    ("talon_truncates_one_short", "npass = room;", "npass = room - 1;", [PINS]),
    ("talon_root_scores_zero", "x->d = 1; x->r[0] = r; x->s = lp[r];", "x->d = 1; x->r[0] = r; x->s = 0.0f;",
     [PINS]),
    ("heap_child_ties_by_larger_rank", "return a < b ? -1 : (a > b ? 1 : 0);", "return a > b ? -1 : (a < b ? 1 : 0);",
     [HEAP]),
    ("heap_first_child_wrong_row", "ch.s = x.s + or_hs_edge(ch.d, c, ord[(size_t)n * K]);",
     "ch.s = x.s + or_hs_edge(ch.d, jpos, ord[(size_t)n * K]);", [HEAP]),
    ("norm_parent_row_off_by_one", "const int u = (d == 0) ? (i == 0 ? root_tok : -1) : id[(d - 1) * K + i];",
     "const int u = (d == 0) ? (i == 0 ? root_tok : -1) : id[d * K + i];", [NORM, HEAP]),
    ("tdes_wrong_depth_row", "a = a + Dd[(int64_t)d * H + h];", "a = a + Dd[(int64_t)(d > 0 ? d - 1 : 0) * H + h];",
     [HEAP]),
    ("saba_hist_over_window", "float hist = n ? (float)sum / (float)n : 0.0f;",
     "float hist = n ? (float)sum / (float)w : 0.0f;", [BUDGETS]),
    ("saba_gain_drops_the_bonus_token", "float a = n ? (float)(sum + n) / (float)n : 1.0f;",
     "float a = n ? (float)sum / (float)n : 1.0f;", [BUDGETS]),
    ("saba_conf_without_exp", "conf += exp((double)top_lp[d]);", "conf += (double)top_lp[d];", [BUDGETS]),
    ("tree_check_skips_depth", "if (depth[n] != depth[p] + 1) return 0;", "", [PINS]),
    ("mask_bit_modulo_31", "row[a / 32] |= 1u << (a % 32);", "row[a / 32] |= 1u << (a % 31);", [PINS]),
    # output assembly: ids, parent indices, ranks, emitted tokens
    ("candidates_write_rank_not_id", "ids[r * Kc + k] = buf[k].id;", "ids[r * Kc + k] = k;", [PINS]),
    ("ddtree_parent_off_by_one", "par = j + 1;", "par = j;", [PINS]),
    ("talon_parent_in_build_order", "parent[i + 1] = x->parent < 0 ? 0 : out_of[x->parent];",
     "parent[i + 1] = x->parent < 0 ? 0 : x->parent + 1;", [PINS]),
    ("talon_score_drops_parent", "x->s = T[v].s + lp[(d - 1) * Kc + w];", "x->s = lp[(d - 1) * Kc + w];", [PINS]),
    ("dartree_parent_supertree_index", "parent[i + 1] = out_of[x->parent];", "parent[i + 1] = x->parent;",
     [PINS, NORM, BUDGETS]),
    ("dartree_rank_of_first_position", "rank[i + 1] = x->r[x->d - 1];\n            score[i + 1] = x->s;\n        }\n"
     "        *n_nodes = n + 1;", "rank[i + 1] = x->r[0];\n            score[i + 1] = x->s;\n        }\n"
     "        *n_nodes = n + 1;", [PINS, NORM, BUDGETS]),
    ("heap_parent_off_by_one", "        parent[n] = p;\n        depth[n] = x.d;\n        rank[n] = c;",
     "        parent[n] = p > 0 ? p - 1 : p;\n        depth[n] = x.d;\n        rank[n] = c;", [HEAP]),
    ("norm_root_token_on_every_row", "const int u = (d == 0) ? (i == 0 ? root_tok : -1) : id[(d - 1) * K + i];",
     "const int u = (d == 0) ? root_tok : id[(d - 1) * K + i];", [NORM, HEAP]),
    ("saba_range_excludes_the_top", "for (int B = B_min; B <= B_max; ++B) {", "for (int B = B_min; B < B_max; ++B) {",
     [BUDGETS]),
    ("positions_from_the_parent", "pos[n] = depth[n] + pos_offset;", "pos[n] = (n ? depth[parent[n]] : 0) + pos_offset;",
     [PINS]),
    ("greedy_emits_last_accepted_token", "*next_tok = a;", "*next_tok = n > 0 ? tok[n] : a;", [PINS]),
    ("t1_no_fallback_to_p_below_children",
     "(drow[v] - lsed));\n                w[v] = P > Q ? P - Q : 0;\n                S += w[v];\n            }\n"
     "        }\n        if (S == 0) {",
     "(drow[v] - lsed));\n                w[v] = P > Q ? P - Q : 0;\n                S += w[v];\n            }\n"
     "        }\n        if (S == 0 && nk == 0) {",
     [PINS]),
]


def _run_pins(lib, files):
    env = dict(os.environ, DT_ORACLE_LIB=lib)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *files]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-3000:]


@pytest.fixture(scope="module")
def outcomes():
    with open(oracle_build.SRC) as f:
        src = f.read()
    os.makedirs(oracle_build.OUT_DIR, exist_ok=True)
    with tempfile.TemporaryDirectory(prefix="mutants_", dir=oracle_build.OUT_DIR) as tmp:
        return _build_and_run(src, tmp)


def _build_and_run(src, tmp):
    jobs = {}
    for name, old, new, files in [("control", None, None, [PINS, BUDGETS, NORM, HEAP, VARIANTS])] + MUTANTS:
        if old is not None:
            assert src.count(old) == 1, "mutant %s: its source text must occur exactly once" % name
            text = src.replace(old, new)
        else:
            text = src
        c_path = os.path.join(tmp, name + ".c")
        with open(c_path, "w") as f:
            f.write(text)
        jobs[name] = (c_path, os.path.join(tmp, "lib" + name + ".so"), files)
    workers = max(2, min(8, os.cpu_count() or 2))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        libs = {n: ex.submit(oracle_build.compile_to, c, so) for n, (c, so, _) in jobs.items()}
        for f in libs.values():
            f.result()
        runs = {n: ex.submit(_run_pins, so, files) for n, (_, so, files) in jobs.items()}
        return {n: f.result() for n, f in runs.items()}


def test_control_build_passes_every_pin(outcomes):
    rc, log = outcomes["control"]
    assert rc == 0, log


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_fails_a_pin(outcomes, name):
    rc, log = outcomes[name]
    # 1: a pin failed; negative: the mutant crashed the child (also caught).
    # Anything else (a usage or collection error) is a broken harness.
    assert rc == 1 or rc < 0, "mutant %s survived the pins (exit %d)\n%s" % (name, rc, log)
