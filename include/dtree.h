/*
 * dtree.h -- C ABI of the draft-tree build / tree-verify library for block
 * (diffusion) drafters, GB300 (sm_103a).
 *
 * One speculative round on the pages: a block drafter scores all L future
 * positions in one pass; per position the library keeps the Top-K tokens and
 * their log-probabilities, selects a budget-B prefix tree (DDTree Top-B,
 * DARTree supertree + deferred Top-B with the Markov correction, plain or
 * normalised over the vocabulary, DARTree's fixed per-depth widths, the
 * best-first heap with Markov or TDES edge scores, or TALON gating; per-request
 * budgets from the caller or from SABA), builds the tree attention mask and
 * position ids, and, once the target model has scored every tree node, walks
 * the longest accepted path (greedy, the T=1 ratio rule, one residual per
 * rejected sibling, target-sample matching, or T=1 against the normalised
 * DARTree proposal).  Sources (by page title):
 *   [DARTree] "DARTree: Speculative Diffusion Decoding With Autoregressive
 *             Draft Trees" -- "Speculative sampling", "Tree verification and
 *             DDTree", Algorithm 1, "Deferred best-first pruning", Lemma 1.
 *   [TALON]   "TALON: Confidence-Aware Speculative Decoding with Adaptive
 *             Token Trees" -- "Key designs" 1 and 2.
 *   [Unit11]  "Sampling, speculative decoding and multi-token prediction"
 *             (formulas-to-systems, unit 11) -- temperature and greedy ties,
 *             the worked three-token example, the bonus token, the >= 1 token
 *             per round argument.
 *   [DDTree]  "DDTree algorithm: efficient inference-tree construction"
 *             (CSDN explainer) -- Prop 1, Prop 2, Lemma (S_K), Algorithm 1
 *             (heap over rank descriptors), section 4.2 (tree attention mask).
 *   [GRAFT]   "GRAFT: adaptive DLM draft-tree construction with
 *             target-distilled edge scoring" -- "Target-distilled edge
 *             scoring", "Inference", "State-aware budget allocation".
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, never synchronises, and enqueues its kernels on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream).
 *  - Arrays are dense, row-major, without padding, laid out as the comment on
 *    each argument says; b = request, L = block positions, V = vocabulary.
 *  - Arguments the host can check (sizes, modes, NULL pointers, limits) are
 *    checked before anything is enqueued: on failure the call returns a
 *    negative dt_status and enqueues nothing.
 *  - Conditions only the device can see (an invalid tree handed to the mask
 *    or verify call, a wait that exceeded its bound) set bits in the caller's
 *    per-request status word (dt_tree.status), readable after the stream
 *    synchronises; see DT_DEV_*.
 *  - A launch failure returns DT_ERR_CUDA (cudaGetLastError is consumed).
 *  - So there are three host error codes: a missing or short workspace is
 *    DT_ERR_INVALID_ARG like any other bad argument, while an invalid tree and
 *    a wait that ran out, which only the device sees, are the status bits
 *    DT_DEV_BAD_TREE and DT_DEV_TIMEOUT rather than return codes.
 *  - dt_tree.rank holds each node's own candidate rank; its full rank
 *    descriptor is the ranks along its parent chain.
 *  - The walk's rules are split over three calls: dt_verify (greedy, or the
 *    T=1 ratio rule with one normalised residual), dt_verify_rule (one
 *    residual per rejected sibling, or target-sample matching) and
 *    dt_verify_markov (T=1 against the normalised DARTree proposal).
 * Limits: L <= 32, V <= DT_MAX_V, candidate list Kc <= 1024, nodes per
 * request (incl. the root) <= 1025.
 */
#ifndef DTREE_H
#define DTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dt_stream_t; /* identical to cudaStream_t */

typedef enum {
    DT_OK = 0,
    DT_ERR_INVALID_ARG = -1, /* a size, mode, limit or pointer is invalid */
    DT_ERR_UNSUPPORTED = -2, /* valid but outside this build's limits */
    DT_ERR_CUDA = -4,        /* a CUDA launch or attribute call failed */
} dt_status;

enum { DT_MODE_DDTREE = 0, DT_MODE_DARTREE = 1, DT_MODE_TALON = 2, DT_MODE_HEAP = 3 };

/* TDES edge scorer ([GRAFT] "Target-distilled edge scoring"):
 *   f(p, c, d) = w . ReLU(W [g_p(e_p); g_c(e_c); e_d] + b) + b0,  term = s * f.
 * The token projections are fixed per token ("computed once and reused"), so
 * the scorer is given by the first layer's per-token and per-depth parts:
 *   Ap[v] = W_p g_p(e_v), Ac[v] = W_c g_c(e_v)  ([V][H] fp32),
 *   Dd[d-1] = W_d e_d + b                         ([L][H] fp32),
 * and per edge, in fp32: a = (Ap[p][h] + Ac[c][h]) + Dd[d-1][h],
 * r = max(a, 0), acc = fma(w[h], r, acc) from 0 over h, term = s * (acc + b0). */
typedef struct {
    int32_t H;          /* hidden units, 1..4096 */
    const float* Ap;    /* [V][H] parent-token rows */
    const float* Ac;    /* [V][H] child-token rows */
    const float* Dd;    /* [L][H] depth rows (bias included) */
    const float* w;     /* [H] output weights */
    float b0;           /* output bias */
    float s;            /* scale */
} dt_tdes;
enum { DT_BF16 = 0, DT_F32 = 1 };

#define DT_MAX_L 32
#define DT_MAX_KC 1024
#define DT_MAX_NODES 1025
#define DT_MAX_V (16 * 32768)

/* Device status word bits (dt_tree.status[b]).  dt_select (and so
 * dt_build_tree) stores a fresh value per request; dt_tree_mask and dt_verify
 * OR their bits into it. */
#define DT_DEV_BAD_TREE 0x1         /* mask/verify: parent/depth arrays invalid */
#define DT_DEV_TIMEOUT 0x2          /* a bounded wait gave up; outputs undefined
                                       (stage 1 marks such a row with a NaN lse,
                                       which dt_select reports with this bit) */
#define DT_DEV_BESTFIRST 0x4        /* DARTree: TopB(S) was not a topologically
                                       ordered tree; the best-first heap over S
                                       was used (see dt_build_tree) */
#define DT_DEV_VIOLATION_SHIFT 8    /* DARTree: number of supertree edges whose
                                       child outscores its parent, saturating
                                       at 2^23-1, in bits 8..30 */

/* Build parameters.  [DARTree] Algorithm 1 inputs (logits, K, W, B, beta);
 * [TALON] settings (root Top-k, mu, node budget N); [DDTree] Algorithm 1
 * (K, budget B).  Budgets count non-root nodes. */
typedef struct {
    int32_t mode;       /* DT_MODE_* */
    int32_t batch;      /* requests b >= 1 */
    int32_t L;          /* block positions, 1..32 */
    int32_t V;          /* vocabulary, >= 1 */
    int32_t dtype;      /* drafter logits: DT_BF16 or DT_F32 */
    int32_t K;          /* DDTree / DARTree: candidates per position, 1..min(V,1024)
                           (DDTree: K = min(B, V) suffices, [DDTree] Lemma (S_K)) */
    int32_t B;          /* DDTree / DARTree node budget, 1..1024 */
    int32_t W;          /* DARTree layer width, 1..1024, W*K <= 4096 */
    float beta;         /* DARTree depth bonus, must be <= 0 ([DARTree] Lemma 1) */
    int32_t R;          /* DARTree Markov rank (columns of U and Vt), 0 = no term */
    const float* U;     /* DARTree [V][R] fp32, parent-token embedding, or NULL */
    const float* Vt;    /* DARTree [V][R] fp32, child-token embedding, or NULL */
    const int32_t* root_tok; /* DARTree [batch] token of the verified prefix's
                           last position (parent of depth-1 nodes), or NULL:
                           no Markov term at depth 1 */
    int32_t talon_k;    /* TALON root-layer Top-k, 1..N */
    float log_mu;       /* TALON log(mu) rounded to fp32, mu in (0, 1] */
    int32_t N;          /* TALON node budget, 1..1024 */
    int32_t markov_norm; /* DARTree (or HEAP with the Markov term) with R > 0:
                           1 = normalise the corrected
                           distribution over the full vocabulary ([DARTree]
                           "Causal correction": q~ is a probability), i.e.
                           log q~ = (lp + <U, Vt>) - log Z_d(parent token),
                           see dt_markov_norm; needs R = 64 and 16-byte
                           aligned U, Vt.  0 = the unnormalised term. */
    const dt_tdes* tdes; /* DT_MODE_HEAP: TDES edge scorer, or NULL (then the
                           Markov term when R > 0, else no edge term) */
    int32_t budget_policy; /* DT_BUDGET_*.  DARTree only: DT_BUDGET_UNIFORM is
                           DARTree (fixed) ([DARTree] experimental setup):
                           depth d keeps B/L children (one more for the first
                           B%L depths), W is ignored, B >= L. */
    const int32_t* budget; /* DDTree and HEAP: [batch] per-request node budgets
                           (e.g. from dt_saba_budget), each clamped to [1, B];
                           NULL: B for every request.  B still sizes the
                           kernels and max_nodes. */
} dt_build_params;
#define DT_BUDGET_TOPB 0
#define DT_BUDGET_UNIFORM 1

/* Tree buffers (caller-owned device memory).  Node 0 of each request is the
 * root (token -1, parent -1, depth 0, rank -1, score 0); nodes 1..n-1 follow
 * in the shared node order: score descending, then rank descriptor ascending
 * (a prefix before its extensions).  Rows n..max_nodes-1 are left untouched. */
typedef struct {
    int32_t max_nodes;  /* row capacity per request, >= budget + 1, <= 1025 */
    int32_t Kc;         /* candidate-list length per position (DDTree/DARTree:
                           K; TALON: min(N, V)) */
    int32_t L;          /* positions (must equal the build's L) */
    int32_t* node_tok;  /* [b][max_nodes] token of each node */
    int32_t* parent;    /* [b][max_nodes] parent node index (root: -1) */
    int32_t* depth;     /* [b][max_nodes] depth (root 0; position = depth) */
    int32_t* rank;      /* [b][max_nodes] 0-based rank of the node's token in
                           its position's candidate list (root -1) */
    float* score;       /* [b][max_nodes] path score (fp32, see each mode) */
    int32_t* n_nodes;   /* [b] nodes including the root */
    float* lse;         /* [b][L] drafter log-normaliser per position */
    int32_t* cand_id;   /* [b][L][Kc] Top-Kc token ids, logit desc, id asc */
    float* cand_lp;     /* [b][L][Kc] their log-probabilities (logit - lse) */
    int32_t* status;    /* [b] DT_DEV_* bits */
} dt_tree;

/* Bytes of caller-provided device workspace dt_build_tree / dt_select need
 * for these parameters (0 for DDTree and TALON; DARTree with R > 0, and HEAP
 * with an edge term: the per-request edge table, batch*L*K*K*4 bytes,
 * rounded up to 256; with
 * markov_norm also the log-normaliser table, batch*L*K*4 bytes rounded up to
 * 256, at byte offset DT_ZNORM_OFFSET(p) = the rounded Markov table size,
 * then scratch for dt_markov_norm).  Returns 0 and sets *ok = 0 on invalid
 * parameters when ok != NULL. */
size_t dt_workspace_size(const dt_build_params* p, int* ok);

/* Stage 1: per-position log-softmax and Top-Kc over the full vocabulary.
 * [DARTree] Algorithm 1 (per-position Top-K); [DDTree] section 3.3 (log-domain scores of the
 * per-position Top-K tokens).
 *   draft_logits: [batch][L][V] in p->dtype (bf16 or fp32); finite values or
 *   -inf (at least one finite value per row).
 * Writes tree->lse [b][L] (fp32 accumulation of sum exp(x - max)),
 * tree->cand_id / cand_lp [b][L][Kc] (rank order: logit descending, token id
 * ascending on equal logits; lp = logit - lse in fp32).  Kc = tree->Kc must be
 * K (DDTree/DARTree) or min(N, V) (TALON).  Does not touch tree->status; a row
 * whose staging wait exceeded its bound gets lse = NaN. */
dt_status dt_candidates(const dt_build_params* p, const void* draft_logits,
                        dt_tree* tree, dt_stream_t stream);

/* Which stage-1 kernel dt_candidates launches for these parameters, without
 * launching anything (a query of the current device's cluster residency may
 * run on the first call).  *kernel = DT_STAGE1_CLUSTER: each row is split over
 * a thread-block cluster of *cluster CTAs (few rows: latency);
 * DT_STAGE1_ROWS: one CTA per row, *cluster = 1 (many rows, or candidate lists
 * longer than 512: throughput).  Returns DT_ERR_INVALID_ARG for parameters
 * dt_candidates would reject on shape (batch, L, V, dtype, Kc). */
#define DT_STAGE1_CLUSTER 1
#define DT_STAGE1_ROWS 2
dt_status dt_stage1_plan(const dt_build_params* p, int32_t* kernel, int32_t* cluster);

/* Measurement kernel, not a step of the method: the read floor of the cluster
 * stage-1 launch.  Reads draft_logits [batch][L][V] with exactly the launch
 * dt_candidates uses when dt_stage1_plan answers DT_STAGE1_CLUSTER (the same
 * clusters, chunks, shared memory and programmatic dependent launch) and does
 * the least work that consumes every byte: each CTA writes its chunk's
 * maximum to chunk_max[row][S] (S = *cluster of dt_stage1_plan; the row
 * maximum is the maximum of a row's S entries).  Its device time is the floor
 * that stage 1's own exchanges and passes add to.  status: NULL, or one int32
 * that gets bit DT_DEV_TIMEOUT (OR-ed) when a staging wait ran out of its bound.
 * Returns DT_ERR_UNSUPPORTED when the plan is DT_STAGE1_ROWS (there the
 * measured HBM copy bandwidth is the floor), DT_ERR_INVALID_ARG as
 * dt_stage1_plan or for a NULL pointer. */
dt_status dt_stage1_ceiling(const dt_build_params* p, const void* draft_logits, float* chunk_max,
                            int32_t* status, dt_stream_t stream);

/* Stages 2-3: tree selection from the candidate lists already in `tree`
 * (written by dt_candidates, or by the caller), writing node_tok, parent,
 * depth, rank, score, n_nodes and a fresh status word per request.
 *  DDTree ([DDTree] Algorithm 1, Prop 2, Lemma (S_K); [DARTree] "Tree
 *   verification and DDTree"): the B best prefixes of S_K under the node
 *   order, score = sum of lp along the path, fp32, added from the root.
 *  DARTree ([DARTree] Algorithm 1, "Deferred best-first pruning", Lemma 1):
 *   per depth, all W*K children of the kept parents scored
 *   s = (s_parent + (lp + <U[tok(parent)], Vt[tok(child)]>)) + beta (the dot
 *   product a serial fp32 fma chain over R; with markov_norm the term is
 *   (lp + <U, Vt>) - log Z from the workspace table that dt_markov_norm, or
 *   the caller, wrote), keep the W best; then TopB over
 *   the supertree S.  When TopB(S) is not a topologically ordered tree (only
 *   possible when some edge raises the score), the result is the best-first
 *   heap over S and DT_DEV_BESTFIRST is set.
 *  TALON ([TALON] key designs 1-2): root layer = Top-talon_k of position 1;
 *   then pool the children of the last layer, keep s >= max_pool + log_mu,
 *   truncate to the best N - |T| and stop on overflow; at most L layers.
 *  HEAP ([DARTree] tree-construction ablation, "sequential correction with
 *   heap"; [GRAFT] "Inference", TDES path scores in a max-heap): best-first
 *   over prefixes with a parent-conditioned edge score
 *   t = lp + E(parent token, child token, depth) (minus log Z with
 *   markov_norm), E the Markov term <U, Vt> (R > 0, tdes NULL), the TDES term
 *   (tdes), or none (then the DDTree result); the children of a parent are
 *   taken in (t desc, rank asc) order, each pop adds the best prefix (score
 *   desc, then its descriptor of order positions) and pushes its first child
 *   and next sibling; B pops.  Nodes are in pop order, parents first; a child
 *   may outscore its parent.  No width limit, unlike DARTree.  Needs K <= 256
 *   and the order tables within shared memory (else DT_ERR_UNSUPPORTED);
 *   dt_select_mask writes the mask with the mask kernel afterwards.
 * workspace: device memory of dt_workspace_size(p) bytes (may be NULL when 0). */
dt_status dt_select(const dt_build_params* p, dt_tree* tree, void* workspace,
                    size_t workspace_bytes, dt_stream_t stream);

/* Full-vocabulary log-normalisers of the corrected DARTree distribution
 * ([DARTree] "Causal correction"), for p->markov_norm = 1.  For every request
 * b, position d and candidate i of position d-1 (the possible parent tokens
 * of depth-(d+1) nodes; at d = 0 the root token, row i = 0 only):
 *   log Z = log sum over every v of exp(lp_d(v) + <U[u], Vt[v]>)
 * written as fp32 to the workspace at DT_ZNORM_OFFSET(p), [b][L][K] (rows
 * without a parent token get 0).  The [b*L*K x 64] x [64 x V] contraction
 * runs on the tensor cores: U and Vt are each split into a bf16 head and a
 * bf16 tail (the rounded remainder) and all four products are accumulated in
 * fp32, so each dot product is within about 2^-17 * sum_k |U[u][k] * Vt[v][k]|
 * of the fp32 tables' and each value within that (at its largest over v) plus
 * the fp32 log-sum-exp's own error (below 1e-5) of the exact one.  Reads
 * draft_logits and tree->cand_id, tree->lse (from dt_candidates).  The
 * workspace must be 16-byte aligned (DT_ERR_INVALID_ARG otherwise).  A row
 * whose bounded wait ran out gets NaN, which dt_select reports as
 * DT_DEV_TIMEOUT. */
#define DT_ZNORM_OFFSET(p) ((((size_t)(p)->batch * (p)->L * (p)->K * (p)->K * 4) + 255) & ~(size_t)255)
dt_status dt_markov_norm(const dt_build_params* p, const void* draft_logits, dt_tree* tree, void* workspace,
                         size_t workspace_bytes, dt_stream_t stream);

/* dt_candidates, then dt_markov_norm when p->markov_norm, then dt_select, on
 * the same stream. */
dt_status dt_build_tree(const dt_build_params* p, const void* draft_logits,
                        dt_tree* tree, void* workspace, size_t workspace_bytes,
                        dt_stream_t stream);

/* dt_select followed by dt_tree_mask: same outputs as the two calls.  For
 * trees of at most 512 rows (max_nodes) the selection kernel writes the mask
 * and positions itself (one kernel launch fewer; its trees have every parent
 * before its children); larger trees get the mask kernel after it.
 * mask/pos as in dt_tree_mask. */
dt_status dt_select_mask(const dt_build_params* p, dt_tree* tree, void* workspace, size_t workspace_bytes,
                         int32_t pos_offset, uint32_t* mask, int32_t* pos, dt_stream_t stream);

/* dt_build_tree followed by dt_tree_mask: dt_candidates, dt_markov_norm when
 * p->markov_norm, then dt_select_mask. */
dt_status dt_build_tree_mask(const dt_build_params* p, const void* draft_logits, dt_tree* tree, void* workspace,
                             size_t workspace_bytes, int32_t pos_offset, uint32_t* mask, int32_t* pos,
                             dt_stream_t stream);

/* Tree-attention ancestor mask and position ids.  [DARTree] "Tree
 * verification and DDTree" (a node attends to the verified context and its
 * root-to-node path); [DDTree] section 4.2.
 *   mask: [batch][max_nodes][ceil(max_nodes/32)] uint32; bit (m % 32) of word
 *         m/32 of row n is 1 iff node m is node n or one of its ancestors;
 *         rows >= n_nodes are not written.
 *   pos:  [batch][max_nodes] int32, pos[n] = depth(n) + pos_offset.
 * Reads tree->parent, depth, n_nodes; a request whose arrays are not a valid
 * tree (root first, parents in range, depth = parent depth + 1 <= L) gets
 * DT_DEV_BAD_TREE and no mask rows. */
dt_status dt_tree_mask(const dt_tree* tree, int32_t batch, int32_t pos_offset,
                       uint32_t* mask, int32_t* pos, dt_stream_t stream);

/* Acceptance walk.  Row n of target_logits is the target model's next-token
 * logits after the path root..n.
 *  temperature 0 ([DARTree] "Speculative sampling"; [Unit11] greedy ties):
 *   at node n take a = argmax of row n (smallest id on ties); descend into the
 *   child of n whose token is a; stop when there is none; emit a.
 *  temperature 1 ([DARTree] "Speculative sampling"; [Unit11] worked example,
 *   bonus token): at node n, test n's children in rank order, child c accepted
 *   iff uniforms[b][0][c] < exp_canon((t_n[c] - lse_t) - (d[c] - lse_d)),
 *   descend into the first accepted one; if all are rejected draw from
 *   max(0, P - Q) (P, Q = floor(2^32 * probability) of the target row of n and
 *   of the drafter row of n's children's position), or from P when that is
 *   empty or n has no children, by inverse CDF with uniforms[b][1][n].
 *   exp_canon is an fp32 exponential by Cody-Waite reduction and a degree-7
 *   Taylor polynomial (one rounding per step), so results are reproducible.
 *   target_logits: [batch][max_nodes][V] (dtype); draft_logits [batch][L][V]
 *   (dtype; T=1 only, else may be NULL); uniforms [batch][2][max_nodes] fp32
 *   in [0,1) (T=1 only).
 *   target_lse: NULL, or [batch][max_nodes] fp32 log-normalisers of the
 *   target rows supplied by the caller (e.g. already computed by the target's
 *   sampler); when NULL the walk computes them (fp32 accumulation) for the rows
 *   it visits.  T=1 only.
 * Outputs: acc_nodes [batch][L+1] (root, then accepted nodes, then -1),
 *   acc_len [batch] (accepted draft tokens), next_tok [batch] (the emitted
 *   correction / bonus token), visited_lse [batch][L+1] (T=1: fp32 target
 *   log-normaliser of each visited row; may be NULL).
 * Uses tree->lse at T=1. */
dt_status dt_verify(const dt_tree* tree, int32_t batch, int32_t V, int32_t dtype,
                    const void* target_logits, const float* target_lse,
                    const void* draft_logits, float temperature, const float* uniforms,
                    int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                    float* visited_lse, dt_stream_t stream);

/* Acceptance walk with an explicit rule.  dt_verify(temperature 0) is
 * DT_VERIFY_GREEDY and dt_verify(temperature 1) is DT_VERIFY_RATIO; the pages
 * state the T=1 rule for one drafted token per position and leave several
 * children per node open, so two more readings are offered:
 *  DT_VERIFY_ITER_RESIDUAL ([Unit11] residual formula applied once per
 *   rejected sibling; [DARTree] "Speculative sampling"): child c_1 of n is
 *   tested as in DT_VERIFY_RATIO; child c_i (i >= 2, rank order) against the
 *   residual r_{i-1} left by rejecting c_1 .. c_{i-1}, r_i = [r_{i-1} - q]_+
 *   normalised, held exactly as the integer weights
 *   W_i = max(0, P - floor(Q * T_i / 2^32)), T_1 = 2^32,
 *   T_{i+1} = T_i + sum_v W_i(v); c_i is accepted iff
 *   floor(u * 2^24) * Q(c_i) * S_{i-1} < W_{i-1}(c_i) * 2^56 (S = sum W).  After
 *   all children are rejected the replacement is drawn from the last residual
 *   (from P when a residual is empty, and then no further child is tested).
 *   With one child per node this is DT_VERIFY_RATIO.  With children drawn
 *   i.i.d. from q it preserves the target distribution; with deterministic
 *   Top-K children neither this nor DT_VERIFY_RATIO is claimed to.  Cost: one
 *   pass over the row per rejected child after the first.
 *  DT_VERIFY_TARGET_MATCH ([DARTree] "Speculative sampling": DFlash's exact
 *   target-sample matching): at each visited node n draw y from P (row n) by
 *   inverse CDF with uniforms[b][1][n]; if a child of n has token y descend
 *   into it, else emit y.  Distribution-preserving for any tree.
 *   draft_logits, tree->lse and uniforms[b][0][*] are not read (draft_logits
 *   may be NULL).
 * Other arguments and outputs as for dt_verify; target_lse and uniforms apply
 * to every T=1 rule.  Returns DT_ERR_INVALID_ARG for an unknown rule. */
/* T=1 walk of a tree built with the normalised DARTree correction
 * ([DARTree] "Causal correction": with the full-vocabulary normaliser the
 * corrected distribution is a probability, so speculative sampling ([DARTree]
 * "Speculative sampling") can test against it).  DT_VERIFY_RATIO's rule with
 * the drafter's proposal of node n's children replaced by
 *   log q~(v | u) = ((d_pos[v] - lse_pos) + <U[u], Vt[v]>) - z,
 * u = tok(n) (the root: p->root_tok[b]), pos = depth(n), z =
 * znorm[b][pos][rank(n)] (the root: znorm[b][0][0]), each step in fp32, the dot
 * product a serial fma chain over R; without a parent token q~ is the plain
 * marginal.  Both the acceptance ratios and the residual max(0, P - Q~) use it.
 * p supplies U, Vt (fp32 [V][R], Vt 16-byte aligned, 4 <= R <= 64, R % 4 == 0),
 * R, root_tok, batch, V, K and dtype; znorm: [batch][L][K] fp32, e.g. the
 * table dt_markov_norm wrote at DT_ZNORM_OFFSET(p).  Other arguments as for
 * dt_verify at temperature 1. */
dt_status dt_verify_markov(const dt_build_params* p, const dt_tree* tree, const void* target_logits,
                           const float* target_lse, const void* draft_logits, const float* znorm,
                           const float* uniforms, int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                           float* visited_lse, dt_stream_t stream);

#define DT_VERIFY_GREEDY 0
#define DT_VERIFY_RATIO 1
#define DT_VERIFY_ITER_RESIDUAL 2
#define DT_VERIFY_TARGET_MATCH 3
dt_status dt_verify_rule(const dt_tree* tree, int32_t batch, int32_t V, int32_t dtype,
                         const void* target_logits, const float* target_lse,
                         const void* draft_logits, int32_t rule, const float* uniforms,
                         int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                         float* visited_lse, dt_stream_t stream);

/* SABA: state-aware per-request budgets ([GRAFT] "State-aware budget
 * allocation").  For every request b, from the candidate tables in `tree`
 * (dt_candidates), optional drafter hidden states and the acceptance history:
 *   1. if prev_acc_len is given and prev_acc_len[b] >= 0, store it in the
 *      ring: ring[b][count[b] % window] = prev_acc_len[b], count[b] += 1;
 *   2. over the last n = min(count[b], window) rounds: hist = (sum l) / n,
 *      a = (sum (l + 1)) / n (fp32; hist = 0, a = 1 with no history);
 *   3. conf = mean over the L positions of exp(lp of the top candidate);
 *      degen = mean of r_d = cos(h_d, h_{d+1}) plus r_{L-2} - r_0 (0 without
 *      hidden states or with L = 1);
 *   4. budget[b] = argmax over the integers B in [B_min, B_max] of
 *      (a * sqrt(B)) / (B * c_verify + c_fixed) in fp32, one rounding per
 *      operation, the smallest B on ties.  As the page prints the model, a
 *      cancels and the optimum is c_fixed / c_verify for every state.
 *   state[b] = (conf, degen, hist, a), fp32.
 * hidden: NULL or [batch][L][Hd] fp32.  ring [batch][window] and count
 * [batch] int32 are caller-owned, zeroed before the first round, updated in
 * place.  budget [batch] int32 feeds dt_build_params.budget.  Returns
 * DT_ERR_INVALID_ARG for window < 1, c_verify <= 0, c_fixed < 0, or B_min,
 * B_max outside 1 <= B_min <= B_max <= 1024. */
typedef struct {
    int32_t window;     /* w: rounds of acceptance history */
    float c_verify;     /* per-node verification cost */
    float c_fixed;      /* fixed per-round cost */
    int32_t B_min;
    int32_t B_max;
} dt_saba_params;
dt_status dt_saba_budget(const dt_saba_params* q, const dt_tree* tree, int32_t batch,
                         const float* hidden, int32_t Hd, const int32_t* prev_acc_len,
                         int32_t* ring, int32_t* count, float* state, int32_t* budget,
                         dt_stream_t stream);

/* Allocation-free DARTree selection.  The pages have no counterpart: this is
 * a service to callers that cannot allocate device memory -- e.g. a serving
 * process whose framework has reserved the whole device budget and lets no
 * library allocate, or a latency-critical path where cudaMalloc/cudaFree are
 * banned because they can synchronise the device.
 * Same result as dt_select with p->mode == DT_MODE_DARTREE, but the Markov
 * table that dt_select keeps in the caller's workspace lives in a fixed array
 * inside the library (DT_NOALLOC_TABLE_BYTES).  CUDA reserves that array on a
 * device when it loads the library's device code there -- under lazy module
 * loading, at the first library call on that device -- and it stays reserved
 * for the life of the device's context.  The caller still owns and passes the
 * tree buffers.  A call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *   - Returns DT_ERR_UNSUPPORTED when batch * L * K * K * 4 exceeds
 *     DT_NOALLOC_TABLE_BYTES or p->markov_norm is set (its normaliser table
 *     needs caller workspace), DT_ERR_INVALID_ARG for a mode other than
 *     DT_MODE_DARTREE, and the usual errors otherwise.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.  The lookup is repeated when the device's context has
 *     changed since (after cudaDeviceReset, for instance); make the first call
 *     after such a change outside stream capture as well.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; each call writes every entry it reads, so none needs clearing.
 *     Calls whose kernels overlap on the GPU (different streams, or
 *     concurrent host threads on one device) race on the array: serialise
 *     them. */
#define DT_NOALLOC_TABLE_BYTES (4u << 20)
dt_status dt_select_dartree_noalloc(const dt_build_params* p, dt_tree* tree, dt_stream_t stream);

/* Test hook of the timeout path (failure detection without a GPU fault).
 * Every mbarrier wait in the library is bounded; when a bound runs out the
 * kernel records it and carries on (stage 1: the row's lse becomes NaN and the
 * selection sets DT_DEV_TIMEOUT; the walk sets DT_DEV_TIMEOUT in the status
 * word; the normaliser writes NaN, which the selection reports the same way).
 * For the kernels named in `kernels` (DT_PROBE_* bits, 0 = off) this makes
 * the staging wait first wait on a barrier that nothing ever completes, bounded
 * by budget_cycles SM clock cycles (1 .. DT_PROBE_MAX_BUDGET), so that path
 * runs; the real wait follows unchanged, so every copy lands before its data
 * is read and outputs other than the flags are the usual ones.  Applies to the
 * current device; synchronous (a copy to device symbols): call it outside
 * stream capture and with no library kernel running.  Not for production use.
 * Returns DT_ERR_INVALID_ARG for unknown bits or a budget out of range. */
#define DT_PROBE_STAGE1 0x1      /* the cluster stage-1 kernel (dt_candidates, few rows) */
#define DT_PROBE_WALK 0x2        /* the acceptance walk (dt_verify, dt_verify_rule, dt_verify_markov) */
#define DT_PROBE_NORMALISER 0x4  /* the tensor-core normaliser (dt_markov_norm) */
#define DT_PROBE_MAX_BUDGET (1ll << 28)
dt_status dt_test_wait_fault(int32_t kernels, int64_t budget_cycles);

/* Static string for a dt_status value. */
const char* dt_status_str(dt_status s);

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t dt_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DTREE_H */
