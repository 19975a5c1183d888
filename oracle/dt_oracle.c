/*
 * dt_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of draft-tree build and tree
 * verification for block (diffusion) drafters.  It exists to check the CUDA
 * path and to serve as the timed CPU baseline; nothing in the product path may
 * call it.  It shares no code, header, table or helper with the CUDA sources.
 *
 * Every function follows one passage of the pages it restates; the page is
 * named by its title and the section, equation or algorithm it falls in:
 *
 *   [DARTree]  "DARTree: Speculative Diffusion Decoding With Autoregressive
 *              Draft Trees" (papercache.org summary).
 *   [TALON]    "TALON: Confidence-Aware Speculative Decoding with Adaptive
 *              Token Trees" (papernotes.org notes).
 *   [Unit11]   "Sampling, speculative decoding and multi-token prediction"
 *              (formulas-to-systems course, unit 11).
 *   [DDTree]   "DDTree algorithm: efficient inference-tree construction"
 *              (CSDN explainer of DDTree).
 *
 * Precision.  The log-normaliser is accumulated in double and rounded once to
 * fp32.  Every quantity that decides an integer result (a tree, an accepted
 * path) is computed in fp32 in a fixed order, because the CUDA path takes those
 * decisions in fp32 too: path scores are added left to right from the root's
 * 0, the DARTree Markov term is a serial fmaf chain from 0.0f, and the T=1
 * acceptance ratio and residual weights use exp_canon (below).  Build with
 * -ffp-contract=off so that no multiply-add is fused behind our back.
 *
 * Parity status of each function is listed in its header comment.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_MAXL 32

enum { OR_OK = 0, OR_EINVAL = -1, OR_ENOMEM = -2, OR_EBADTREE = -5 };

/* ------------------------------------------------------------------------- */
/* exp_canon: fp32 exponential by Cody and Waite's argument reduction          */
/* (W. J. Cody, W. Waite, "Software Manual for the Elementary Functions",      */
/* 1980): x = k ln2 + r with ln 2 split into a head whose product with k is    */
/* exact and a tail, then e^r by its Taylor series to degree 7 in Horner form, */
/* then scaling by 2^k.  Every step is one correctly rounded fp32 operation,   */
/* so any IEEE machine with a true fma produces the same bits.                 */
/* Range: returns 0 for x < -86 (results below 2^-124) and +inf for x > 88.5;  */
/* every x <= 88.5 gives a finite value (e^88.5 < FLT_MAX).  Near the top k    */
/* reaches 128, whose 2^k is not a float, so 2^k is applied as 2^127 * 2:      */
/* both are exact scalings, so the product is rounded once, as for smaller k.  */
/* Pinned: ulp error against double exp, monotonicity (tests).                 */
/* ------------------------------------------------------------------------- */
static float or_pow2i(int k) /* 2^k for -126 <= k <= 127, built from its bits */
{
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)(k + 127) << 23;
    return v.f;
}

float or_exp_canon(float x)
{
    const float log2e = 1.44269504088896340736f;
    const float ln2_hi = 0.693145751953125f;        /* 16 significant bits */
    const float ln2_lo = 1.42860682030941723212e-6f; /* ln2 - ln2_hi */
    if (x != x) return x;
    if (x > 88.5f) return INFINITY;
    if (x < -86.0f) return 0.0f;
    float t = x * log2e;
    float kf = rintf(t);
    int k = (int)kf;
    float r = fmaf(-kf, ln2_hi, x);
    r = fmaf(-kf, ln2_lo, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    if (k > 127) return (p * or_pow2i(127)) * 2.0f;
    return p * or_pow2i(k);
}

void or_exp_canon_vec(const float* x, int64_t n, float* y)
{
    for (int64_t i = 0; i < n; ++i) y[i] = or_exp_canon(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Stage 1: per-position log-softmax and Top-Kc candidate list.                */
/* [DARTree] Algorithm 1, its per-position Top-K candidate step; [DDTree]      */
/* section 3.3 (scores are log-probabilities of the per-position Top-K tokens).*/
/* Rank order: logit descending, token id ascending on equal logits.           */
/* lse = max + log(sum exp(x - max)) in double, rounded once to fp32;          */
/* lp = x - lse in fp32.                                                       */
/* Pinned: closed forms (uniform row, shift invariance), sum of exp(lp) = 1,   */
/* brute-force sort in the tests.                                              */
/* ------------------------------------------------------------------------- */
typedef struct { float v; int32_t id; } or_vi;

static int or_cmp_vi(const void* pa, const void* pb)
{
    const or_vi* a = (const or_vi*)pa;
    const or_vi* b = (const or_vi*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

int or_candidates(const float* x, int64_t rows, int32_t V, int32_t Kc,
                  double* lse64, float* lse32, int32_t* ids, float* lps)
{
    if (V < 1 || Kc < 1 || Kc > V) return OR_EINVAL;
    or_vi* buf = (or_vi*)malloc((size_t)V * sizeof(or_vi));
    if (!buf) return OR_ENOMEM;
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = x + r * (int64_t)V;
        double m = -INFINITY;
        for (int32_t v = 0; v < V; ++v)
            if ((double)row[v] > m) m = (double)row[v];
        double s = 0.0;
        if (m != -INFINITY)
            for (int32_t v = 0; v < V; ++v) s += exp((double)row[v] - m);
        double l = (m == -INFINITY) ? m : m + log(s);
        float l32 = (float)l;
        if (lse64) lse64[r] = l;
        lse32[r] = l32;
        for (int32_t v = 0; v < V; ++v) { buf[v].v = row[v]; buf[v].id = v; }
        qsort(buf, (size_t)V, sizeof(or_vi), or_cmp_vi);
        for (int32_t k = 0; k < Kc; ++k) {
            float lp = buf[k].v - l32;
            ids[r * Kc + k] = buf[k].id;
            lps[r * Kc + k] = lp;
        }
    }
    free(buf);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Total order on tree nodes shared by all selections below: higher score      */
/* first; on equal scores, the lexicographically smaller rank descriptor       */
/* (0-based per-position ranks), a proper prefix before its extensions.        */
/* [DARTree] Lemma 1 ("ancestors first on ties"); [DDTree] section 3.3 (heap   */
/* of (-score, rho) tuples orders equal scores by the descriptor tuple).       */
/* Pinned: a parent and child of equal score (lp = 0) stay in that order in    */
/* TALON's output and in DARTree's TopB(S) (tests).                            */
/* ------------------------------------------------------------------------- */
typedef struct {
    float s;               /* path score */
    int32_t d;             /* depth (1-based position of the last token) */
    int32_t r[OR_MAXL];    /* rank descriptor rho_1..rho_d, 0-based */
    int32_t tok;           /* token of the last position */
    int32_t parent;        /* index of the parent in the caller's node list */
    int32_t self;          /* caller-side index */
} or_node;

static int or_lex_less(const int32_t* a, int da, const int32_t* b, int db)
{
    int n = da < db ? da : db;
    for (int i = 0; i < n; ++i)
        if (a[i] != b[i]) return a[i] < b[i];
    return da < db;
}

static int or_before(const or_node* a, const or_node* b)
{
    if (a->s > b->s) return 1;
    if (a->s < b->s) return 0;
    return or_lex_less(a->r, a->d, b->r, b->d);
}

static int or_cmp_node(const void* pa, const void* pb)
{
    const or_node* a = (const or_node*)pa;
    const or_node* b = (const or_node*)pb;
    if (or_before(a, b)) return -1;
    if (or_before(b, a)) return 1;
    return 0;
}

/* A plain binary max-heap under or_before. */
typedef struct { or_node* a; int n, cap; } or_heap;

static int or_heap_push(or_heap* h, const or_node* x)
{
    if (h->n == h->cap) {
        int nc = h->cap ? 2 * h->cap : 64;
        or_node* na = (or_node*)realloc(h->a, (size_t)nc * sizeof(or_node));
        if (!na) return OR_ENOMEM;
        h->a = na; h->cap = nc;
    }
    int i = h->n++;
    h->a[i] = *x;
    while (i > 0) {
        int p = (i - 1) / 2;
        if (!or_before(&h->a[i], &h->a[p])) break;
        or_node t = h->a[i]; h->a[i] = h->a[p]; h->a[p] = t;
        i = p;
    }
    return OR_OK;
}

static or_node or_heap_pop(or_heap* h)
{
    or_node top = h->a[0];
    h->a[0] = h->a[--h->n];
    int i = 0;
    for (;;) {
        int l = 2 * i + 1, r = l + 1, b = i;
        if (l < h->n && or_before(&h->a[l], &h->a[b])) b = l;
        if (r < h->n && or_before(&h->a[r], &h->a[b])) b = r;
        if (b == i) break;
        or_node t = h->a[i]; h->a[i] = h->a[b]; h->a[b] = t;
        i = b;
    }
    return top;
}

/* Tree output arrays, node 0 = root (token -1, parent -1, depth 0, rank -1,
 * score 0). */
typedef struct {
    int32_t* tok; int32_t* parent; int32_t* depth; int32_t* rank; float* score;
} or_tree_out;

static void or_put_root(or_tree_out* o)
{
    o->tok[0] = -1; o->parent[0] = -1; o->depth[0] = 0; o->rank[0] = -1;
    o->score[0] = 0.0f;
}

/* ------------------------------------------------------------------------- */
/* DDTree Top-B by the best-first heap over rank descriptors.                  */
/* [DDTree] section 3.1 (Algorithm 1: start from (1), pop the best descriptor, */
/* add it to the tree, push its first child and its next sibling, stop at B    */
/* nodes), section 3.3 (log-domain scores, first child only below the depth    */
/* cap, next sibling only while rho_d < K); [DARTree] "Tree verification and   */
/* DDTree" (heap best-first, O(B log B)).                                      */
/*                                                                             */
/* The printed successor rule pushes the first child only when rho_d is the   */
/* top rank, which leaves (2,1) unreachable, against the same section's claim  */
/* that every prefix of S_K is reached through pred().  rule = 0 (the reading  */
/* used everywhere) pushes the first child of every popped node; rule = 1      */
/* keeps the printed condition and exists only so that a test can show the    */
/* brute-force pin rejects it.                                                 */
/* Score of (rho_1..rho_d) = lp_1[rho_1] + ... + lp_d[rho_d], fp32, left to    */
/* right from 0.  B counts non-root nodes.                                     */
/* Pinned: brute-force enumeration of S_K (tests), prefix closure, objective   */
/* optimality on tiny vocabularies.                                            */
/* ------------------------------------------------------------------------- */
static float or_desc_score(const float* lp, int K, const int32_t* r, int d)
{
    float s = 0.0f;
    for (int i = 0; i < d; ++i) s = s + lp[i * K + r[i]];
    return s;
}

int or_ddtree(const float* lp, const int32_t* id, int L, int K, int B, int rule,
              int Mmax, int32_t* tok, int32_t* parent, int32_t* depth,
              int32_t* rank, float* score, int32_t* n_nodes)
{
    if (L < 1 || L > OR_MAXL || K < 1 || B < 1 || Mmax < 1) return OR_EINVAL;
    or_tree_out o = { tok, parent, depth, rank, score };
    or_put_root(&o);
    or_node* popped = (or_node*)calloc((size_t)B + 1, sizeof(or_node));
    or_heap h = { 0, 0, 0 };
    if (!popped) return OR_ENOMEM;
    or_node first;
    memset(&first, 0, sizeof first);
    first.d = 1; first.r[0] = 0; first.s = or_desc_score(lp, K, first.r, 1);
    int rc = or_heap_push(&h, &first);
    int n = 0;
    while (rc == OR_OK && n < B && h.n > 0) {
        or_node x = or_heap_pop(&h);
        /* the parent is the popped node whose descriptor is x's minus its last rank */
        int par = 0;
        if (x.d > 1) {
            par = -1;
            for (int j = 0; j < n && par < 0; ++j)
                if (popped[j].d == x.d - 1 &&
                    memcmp(popped[j].r, x.r, sizeof(int32_t) * (size_t)(x.d - 1)) == 0)
                    par = j + 1;
            if (par < 0) { rc = OR_EINVAL; break; }
        }
        popped[n] = x;
        ++n;
        if (n >= Mmax) { rc = OR_EINVAL; break; }
        tok[n] = id[(x.d - 1) * K + x.r[x.d - 1]];
        parent[n] = par;
        depth[n] = x.d;
        rank[n] = x.r[x.d - 1];
        score[n] = x.s;
        int push_child = (x.d < L) && (rule == 0 || x.r[x.d - 1] == 0);
        if (push_child) {
            or_node c = x;
            c.r[c.d] = 0; c.d += 1;
            c.s = or_desc_score(lp, K, c.r, c.d);
            rc = or_heap_push(&h, &c);
        }
        if (rc == OR_OK && x.r[x.d - 1] + 1 < K) {
            or_node sib = x;
            sib.r[sib.d - 1] += 1;
            sib.s = or_desc_score(lp, K, sib.r, sib.d);
            rc = or_heap_push(&h, &sib);
        }
    }
    *n_nodes = n + 1;
    free(popped);
    free(h.a);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* DARTree depth-wise supertree and deferred pruning.                          */
/* [DARTree] Algorithm 1 (depth-wise construction, then pruning) and the       */
/* equation for s_beta in "Deferred best-first pruning"; Lemma 1 and proof.    */
/*                                                                             */
/* The correction head g is a parent-conditioned Markov term on the top-K      */
/* candidates: log q~_d(c | u) = lp_d(c) + <U[tok(u)], Vt[c]>, the dot product */
/* a serial fmaf chain over R terms from 0.0f; at depth 1 the parent is the    */
/* root, whose token is root_tok (no term when root_tok < 0).                  */
/* Child score, in the algorithm's order: (s(parent) + log q~) + beta.         */
/* widths (optional) gives each depth its own width, e.g. DARTree (fixed)'s    */
/* uniform per-depth budget (or_uniform_widths).                               */
/* Each depth keeps the W best children of all parents (shared node order).   */
/* The final pruning takes T = TopB(S).  Lemma 1 proves TopB(S) equals the     */
/* best-first heap over S when beta <= 0 and every log q~ <= 0.  This returns  */
/* the best-first heap result (always a prefix-closed tree) and reports via    */
/* info whether it equals TopB(S) in content and order:                        */
/*   info[0] = 1 if BestFirst_B(S) == TopB(S) (same nodes, same order)         */
/*   info[1] = number of edges of S whose child outscores its parent           */
/*   info[2] = |S| (non-root supertree nodes)                                  */
/* With znorm (the full-vocabulary normalised correction, or_markov_norm):     */
/* log q~ = (lp + <U, Vt>) - log Z, every term rounded to fp32 in that order.   */
/* Pinned: reduction to the DDTree heap for U = 0, beta = 0 and W wide enough  */
/* to keep every prefix; Lemma 1 equality; a beta > 0 counterexample (tests).  */
/* ------------------------------------------------------------------------- */
static float or_markov(const float* U, const float* Vt, int R, int p, int c)
{
    float acc = 0.0f;
    for (int k = 0; k < R; ++k)
        acc = fmaf(U[(int64_t)p * R + k], Vt[(int64_t)c * R + k], acc);
    return acc;
}

int or_dartree(const float* lp, const int32_t* id, int L, int K,
               const float* U, const float* Vt, int R, int root_tok,
               const float* znorm /* nullable [L][K]: log-normalisers, see or_markov_norm */,
               int W, const int32_t* widths /* nullable [L]: width of each depth (<= W) */,
               float beta, int B, int Mmax,
               int32_t* tok, int32_t* parent, int32_t* depth, int32_t* rank,
               float* score, int32_t* n_nodes, int32_t* info,
               int32_t* topb_out /* nullable [Mmax]: TopB(S) as supertree indices */)
{
    if (L < 1 || L > OR_MAXL || K < 1 || W < 1 || B < 1 || Mmax < 1) return OR_EINVAL;
    if (widths)
        for (int d = 0; d < L; ++d)
            if (widths[d] < 1 || widths[d] > W) return OR_EINVAL;
    if ((U == NULL) != (Vt == NULL)) return OR_EINVAL;
    int cap = 1 + W * L;
    or_node* S = (or_node*)calloc((size_t)cap, sizeof(or_node)); /* S[0] = root */
    or_node* kids = (or_node*)calloc((size_t)W * K + K, sizeof(or_node));
    if (!S || !kids) { free(S); free(kids); return OR_ENOMEM; }
    S[0].s = 0.0f; S[0].d = 0; S[0].tok = root_tok; S[0].parent = -1; S[0].self = 0;
    int nS = 1, prev_lo = 0, prev_hi = 1;
    for (int d = 1; d <= L; ++d) {
        int nk = 0;
        for (int p = prev_lo; p < prev_hi; ++p) {
            for (int j = 0; j < K; ++j) {
                int c = id[(d - 1) * K + j];
                float l = lp[(d - 1) * K + j];
                float t;
                int ptok = S[p].tok;
                if (U != NULL && ptok >= 0) {
                    t = l + or_markov(U, Vt, R, ptok, c);
                    /* normalised correction: minus log Z of the parent's row,
                     * row (position d-1, parent's rank at position d-2), or
                     * row (0, 0) for the root */
                    if (znorm != NULL) t = t - znorm[(d - 1) * K + (d == 1 ? 0 : S[p].r[d - 2])];
                } else {
                    t = l;
                }
                or_node* x = &kids[nk++];
                *x = S[p];
                x->r[d - 1] = j;
                x->d = d;
                x->s = (S[p].s + t) + beta;
                x->tok = c;
                x->parent = p;
            }
        }
        qsort(kids, (size_t)nk, sizeof(or_node), or_cmp_node);
        int Wd = widths ? widths[d - 1] : W;
        int keep = nk < Wd ? nk : Wd;
        prev_lo = nS;
        for (int i = 0; i < keep; ++i) { S[nS] = kids[i]; S[nS].self = nS; ++nS; }
        prev_hi = nS;
    }
    int nsup = nS - 1;
    int viol = 0;
    for (int i = 1; i < nS; ++i)
        if (S[i].s > S[S[i].parent].s) ++viol;

    /* TopB(S), the deferred pruning */
    or_node* sorted = (or_node*)malloc((size_t)nsup * sizeof(or_node));
    memcpy(sorted, S + 1, (size_t)nsup * sizeof(or_node));
    qsort(sorted, (size_t)nsup, sizeof(or_node), or_cmp_node);
    int nb = nsup < B ? nsup : B;

    /* BestFirst_B(S): heap from the root's children, push the popped node's
     * children in S, stop after B pops. */
    or_heap h = { 0, 0, 0 };
    int* out_of = (int*)malloc((size_t)nS * sizeof(int));
    int32_t* order = (int32_t*)malloc((size_t)(nb + 1) * sizeof(int32_t));
    int rc = OR_OK;
    for (int i = 0; i < nS; ++i) out_of[i] = -1;
    out_of[0] = 0;
    for (int i = 1; i < nS && rc == OR_OK; ++i)
        if (S[i].parent == 0) rc = or_heap_push(&h, &S[i]);
    int n = 0;
    while (rc == OR_OK && n < B && h.n > 0) {
        or_node x = or_heap_pop(&h);
        order[n++] = x.self;
        out_of[x.self] = n;
        for (int i = 1; i < nS && rc == OR_OK; ++i)
            if (S[i].parent == x.self) rc = or_heap_push(&h, &S[i]);
    }
    if (n + 1 > Mmax) rc = OR_EINVAL;
    if (rc == OR_OK) {
        or_tree_out o = { tok, parent, depth, rank, score };
        or_put_root(&o);
        for (int i = 0; i < n; ++i) {
            const or_node* x = &S[order[i]];
            tok[i + 1] = x->tok;
            parent[i + 1] = out_of[x->parent];
            depth[i + 1] = x->d;
            rank[i + 1] = x->r[x->d - 1];
            score[i + 1] = x->s;
        }
        *n_nodes = n + 1;
        int same = (n == nb);
        for (int i = 0; same && i < n; ++i) same = (sorted[i].self == order[i]);
        info[0] = same;
        info[1] = viol;
        info[2] = nsup;
        if (topb_out)
            for (int i = 0; i < nb && i + 1 < Mmax; ++i) topb_out[i] = sorted[i].self;
    }
    free(h.a); free(out_of); free(order); free(sorted); free(S); free(kids);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* DARTree (fixed): the node budget spread uniformly over the depths.          */
/* [DARTree] experimental setup: the fixed variant allots the budget evenly to */
/* the 16 depths (4 nodes per layer for B = 64).  When L does not divide B the */
/* remainder goes one node each to the shallowest depths (nearest the root,    */
/* the likeliest to be accepted).  The widths feed or_dartree; their sum is B, */
/* so the deferred pruning keeps the whole supertree.                          */
/* Pinned: B = 64, L = 16 gives 4 per layer (the page's figure); sums and      */
/* spreads of every (B, L) (tests).                                            */
/* ------------------------------------------------------------------------- */
int or_uniform_widths(int B, int L, int32_t* widths)
{
    if (B < L || L < 1) return OR_EINVAL;
    for (int d = 0; d < L; ++d) widths[d] = B / L + (d < B % L ? 1 : 0);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* SABA: state-aware budget allocation.                                        */
/* [GRAFT] "State-aware budget allocation": the state s_t = [conf, degen,      */
/* hist] with conf = mean over the D positions of the drafter's probability of */
/* its top candidate, hist = mean acceptance over the last w rounds, degen =   */
/* mean of the adjacent-position cosine similarities r_d = cos(h_d, h_{d+1})   */
/* of the drafter's hidden states plus their growth r_{D-1} - r_1; gain        */
/* G(B) = a * B^beta with beta = 0.5 and a = mean of (l + 1) over the last w   */
/* accepted lengths l; cost C(B) = B * c_verify + c_fixed; B_t = argmax G / C. */
/* As printed, a scales G and cancels in the argmax, which is therefore        */
/* c_fixed / c_verify for every state (beta = 0.5; flagged, not repaired).     */
/* Readings: hist and a use the rounds recorded so far when fewer than w       */
/* (hist = 0, a = 1 with none); the argmax runs over the integers              */
/* [B_min, B_max], the smallest B on ties, with U(B) evaluated in fp32 as      */
/* (a * sqrtf(B)) / (B * c_verify + c_fixed), one rounding per operation.      */
/* The history ring: before the state is read, prev_len (if >= 0) is stored at */
/* ring[count % w] and count is incremented.  conf, degen in double.           */
/* Pinned: argmax = c_fixed / c_verify when that is an integer in range, the    */
/* clamps, independence from the history, hand-computed conf / degen / hist /  */
/* a, the smallest of budgets whose fp32 scores tie (tests).                   */
/* ------------------------------------------------------------------------- */
int or_saba(const float* top_lp /* [D] lp of each position's top candidate */, int D,
            const float* hidden /* nullable [D][Hd] */, int Hd,
            int32_t* ring /* [w] */, int32_t* count, int w, int prev_len,
            float c_verify, float c_fixed, int B_min, int B_max,
            float* state /* [4]: conf, degen, hist, a */, int32_t* budget)
{
    if (D < 1 || w < 1 || B_min < 1 || B_max < B_min || !(c_verify > 0.0f) || !(c_fixed >= 0.0f)) return OR_EINVAL;
    if (prev_len >= 0) { ring[*count % w] = prev_len; *count += 1; }
    int n = *count < w ? *count : w;
    int64_t sum = 0;
    for (int i = 0; i < n; ++i) sum += ring[(*count - 1 - i) % w];
    float hist = n ? (float)sum / (float)n : 0.0f;
    float a = n ? (float)(sum + n) / (float)n : 1.0f;
    double conf = 0.0;
    for (int d = 0; d < D; ++d) conf += exp((double)top_lp[d]);
    conf /= D;
    double degen = 0.0;
    if (hidden && D >= 2) {
        double r0 = 0.0, rl = 0.0, rs = 0.0;
        for (int d = 0; d + 1 < D; ++d) {
            double dot = 0.0, n1 = 0.0, n2 = 0.0;
            for (int k = 0; k < Hd; ++k) {
                double x = hidden[(int64_t)d * Hd + k], y = hidden[(int64_t)(d + 1) * Hd + k];
                dot += x * y; n1 += x * x; n2 += y * y;
            }
            double r = (n1 > 0.0 && n2 > 0.0) ? dot / sqrt(n1 * n2) : 0.0;
            if (d == 0) r0 = r;
            rl = r;
            rs += r;
        }
        degen = rs / (D - 1) + (rl - r0);
    }
    int best = B_min;
    float bu = -1.0f;
    for (int B = B_min; B <= B_max; ++B) {
        float u = (a * sqrtf((float)B)) / ((float)B * c_verify + c_fixed);
        if (u > bu) { bu = u; best = B; }
    }
    state[0] = (float)conf; state[1] = (float)degen; state[2] = hist; state[3] = a;
    *budget = best;
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Full-vocabulary normaliser of the corrected drafter distribution.           */
/* [DARTree] "Causal correction": q~ is a probability over the vocabulary, so  */
/* q~_d(v | u) = exp(lp_d(v) + <U[u], Vt[v]>) / Z_d(u) with                      */
/* Z_d(u) = sum over every v of exp(lp_d(v) + <U[u], Vt[v]>).                     */
/* Row (d, i) of z (0-based position d, i < K) holds log Z_d(u) for the parent  */
/* token u of depth-(d+1) children: the i-th candidate of position d-1, or the  */
/* root token at d = 0 (row (0, 0) only; the other rows of position 0, and all */
/* of them when root_tok < 0, have no term and hold 0).                         */
/* In double: lse_d = log sum_v exp x_d(v); lp_d(v) = x_d(v) - lse_d; the dot    */
/* product; log Z = a_max + log sum_v exp(a_v - a_max).  Rounded once to fp32.  */
/* only_row >= 0 computes that flat row (d * K + i) alone and leaves the rest. */
/* Test infrastructure.                                                        */
/* Pinned: U = 0 gives 0; one token gives its own term; hand-computed V = 3    */
/* golden case; a constant added to every term shifts it; the normalised      */
/* terms sum to 1; bounds max a <= log Z <= max a + log V (tests).             */
/* ------------------------------------------------------------------------- */
int or_markov_norm(const float* x /* [L][V] */, int L, int V, const int32_t* id /* [L][K] */, int K,
                   const float* U, const float* Vt, int R, int root_tok, int only_row,
                   float* z /* [L][K] */)
{
    if (L < 1 || L > OR_MAXL || V < 1 || K < 1 || R < 0 || !x || !id || !U || !Vt || !z) return OR_EINVAL;
    double* a = (double*)malloc((size_t)V * sizeof(double));
    if (!a) return OR_ENOMEM;
    for (int d = 0; d < L; ++d) {
        const float* xd = x + (int64_t)d * V;
        int need = 0;
        for (int i = 0; i < K; ++i) need |= (only_row < 0 || only_row == d * K + i);
        if (!need) continue;
        double mx = -INFINITY;
        for (int v = 0; v < V; ++v) if ((double)xd[v] > mx) mx = (double)xd[v];
        double sx = 0.0;
        for (int v = 0; v < V; ++v) sx += exp((double)xd[v] - mx);
        const double lse = mx + log(sx);
        for (int i = 0; i < K; ++i) {
            if (only_row >= 0 && only_row != d * K + i) continue;
            const int u = (d == 0) ? (i == 0 ? root_tok : -1) : id[(d - 1) * K + i];
            if (u < 0) { z[d * K + i] = 0.0f; continue; }
            double am = -INFINITY;
            for (int v = 0; v < V; ++v) {
                double m = 0.0;
                for (int k = 0; k < R; ++k) m += (double)U[(int64_t)u * R + k] * (double)Vt[(int64_t)v * R + k];
                a[v] = ((double)xd[v] - lse) + m;
                if (a[v] > am) am = a[v];
            }
            double sa = 0.0;
            for (int v = 0; v < V; ++v) sa += exp(a[v] - am);
            z[d * K + i] = (float)(am + log(sa));
        }
    }
    free(a);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Parent-conditioned edge terms on the candidate lattice.                     */
/* E[d][i][j] is the term of the edge from candidate i of position d-1 (the    */
/* parent's token) to candidate j of position d; row 0 of position 0 belongs   */
/* to the root, whose token is root_tok (all zeros when root_tok < 0: no term). */
/* or_markov_table: [DARTree] "Causal correction" (Markov head <U[p], Vt[c]>), */
/* the serial fmaf chain of or_markov.                                         */
/* or_tdes_table: [GRAFT] "Target-distilled edge scoring", the edge scorer     */
/* f(p, c, d) = w . ReLU(W [g_p(e_p); g_c(e_c); e_d] + b) + b0 with its        */
/* learned scale s.  The projections depend on the token only ("computed once  */
/* and reused"), and so does the first layer's product with them, so the       */
/* inputs are the per-token rows Ap[v] = W_p g_p(e_v), Ac[v] = W_c g_c(e_v)    */
/* ([V][H]) and the per-depth row Dd[d-1] = W_d e_d + b ([L][H]).  In fp32:     */
/* a = (Ap[p][h] + Ac[c][h]) + Dd[d-1][h], r = max(a, 0), acc = fmaf(w[h], r,  */
/* acc) from 0 over h, E = s * (acc + b0).  The edge score of the tree builder */
/* is then lp + E (the page's training target softmax(log q + f) and its      */
/* inference path score, a sum of edge scores).                               */
/* Pinned: hand-computed two-unit edges, the ReLU cut, a float64 restatement   */
/* within rounding (tests).                                                    */
/* ------------------------------------------------------------------------- */
int or_markov_table(const int32_t* id, int L, int K, const float* U, const float* Vt, int R, int root_tok,
                    float* E /* [L][K][K] */)
{
    if (L < 1 || L > OR_MAXL || K < 1 || R < 1 || !U || !Vt || !E) return OR_EINVAL;
    memset(E, 0, sizeof(float) * (size_t)L * K * K);
    for (int d = 0; d < L; ++d) {
        int np = d == 0 ? (root_tok >= 0 ? 1 : 0) : K;
        for (int i = 0; i < np; ++i) {
            int ptok = d == 0 ? root_tok : id[(d - 1) * K + i];
            for (int j = 0; j < K; ++j)
                E[((int64_t)d * K + i) * K + j] = or_markov(U, Vt, R, ptok, id[d * K + j]);
        }
    }
    return OR_OK;
}

int or_tdes_table(const int32_t* id, int L, int K, const float* Ap, const float* Ac, const float* Dd,
                  const float* w, int H, float b0, float s, int root_tok, float* E /* [L][K][K] */)
{
    if (L < 1 || L > OR_MAXL || K < 1 || H < 1 || !Ap || !Ac || !Dd || !w || !E) return OR_EINVAL;
    memset(E, 0, sizeof(float) * (size_t)L * K * K);
    for (int d = 0; d < L; ++d) {
        int np = d == 0 ? (root_tok >= 0 ? 1 : 0) : K;
        for (int i = 0; i < np; ++i) {
            int ptok = d == 0 ? root_tok : id[(d - 1) * K + i];
            for (int j = 0; j < K; ++j) {
                int ctok = id[d * K + j];
                float acc = 0.0f;
                for (int h = 0; h < H; ++h) {
                    float a = Ap[(int64_t)ptok * H + h] + Ac[(int64_t)ctok * H + h];
                    a = a + Dd[(int64_t)d * H + h];
                    float r = a > 0.0f ? a : 0.0f;
                    acc = fmaf(w[h], r, acc);
                }
                E[((int64_t)d * K + i) * K + j] = s * (acc + b0);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Best-first heap with parent-conditioned edge scores.                        */
/* [DARTree] tree-construction ablation (Table 2): "sequential correction with */
/* heap" alternates the correction of a popped node's children with heap      */
/* updates; [GRAFT] "Inference": prefixes ordered in a max-heap by the sum of  */
/* their edge scores, the best one added to the tree until the budget is met. */
/* Edge score of child j (position d) under parent u (candidate i of position  */
/* d-1, or the root at d = 1): t = lp_d[j] + E[d-1][i][j], then minus           */
/* znorm[d-1][i] when given (the normalised DARTree correction), in fp32; the   */
/* path score adds t to the parent's score.  The children of u in the order    */
/* (t desc, j asc) play the part of DDTree's ranks: each pop adds the node,    */
/* pushes its first child (below depth L) and its next sibling in its parent's */
/* order.  Heap order: score desc, then the descriptor of order positions      */
/* lexicographically (a prefix first), as in or_ddtree.  Nodes are output in   */
/* pop order (parents before children); rank = the node's candidate rank.     */
/* B counts non-root nodes.  With E = NULL (and no znorm) this is or_ddtree.   */
/* Pinned: reduction to or_ddtree, brute force over every prefix of tiny       */
/* lattices with non-positive edge scores, the best-first invariant with       */
/* arbitrary signs, and DARTree without width pruning (tests).                 */
/* ------------------------------------------------------------------------- */
/* The comparator's context, one copy per thread: callers may run several
 * heaps at once on host threads. */
static _Thread_local const float* or_hs_lp;
static _Thread_local const float* or_hs_E;
static _Thread_local const float* or_hs_z;
static _Thread_local int or_hs_K, or_hs_i, or_hs_d;

static float or_hs_edge(int d, int i, int j) /* d: 1-based position of the child */
{
    int K = or_hs_K;
    float t = or_hs_lp[(d - 1) * K + j];
    if (or_hs_E) t = t + or_hs_E[((int64_t)(d - 1) * K + i) * K + j];
    if (or_hs_z) t = t - or_hs_z[(d - 1) * K + i];
    return t;
}

static int or_hs_cmp(const void* pa, const void* pb)
{
    int a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    float ta = or_hs_edge(or_hs_d, or_hs_i, a), tb = or_hs_edge(or_hs_d, or_hs_i, b);
    if (ta > tb) return -1;
    if (ta < tb) return 1;
    return a < b ? -1 : (a > b ? 1 : 0);
}

/* the children of candidate i of position d-1 (i = 0 for the root at d = 1) in edge order */
static void or_hs_order(int d, int i, int K, int32_t* ord)
{
    for (int j = 0; j < K; ++j) ord[j] = j;
    or_hs_d = d; or_hs_i = i; or_hs_K = K;
    qsort(ord, (size_t)K, sizeof(int32_t), or_hs_cmp);
}

int or_heap_select(const float* lp, const int32_t* id, int L, int K,
                   const float* E /* nullable [L][K][K] */, const float* znorm /* nullable [L][K] */,
                   int B, int Mmax, int32_t* tok, int32_t* parent, int32_t* depth,
                   int32_t* rank, float* score, int32_t* n_nodes)
{
    if (L < 1 || L > OR_MAXL || K < 1 || B < 1 || Mmax < 1) return OR_EINVAL;
    or_tree_out o = { tok, parent, depth, rank, score };
    or_put_root(&o);
    or_hs_lp = lp; or_hs_E = E; or_hs_z = znorm; or_hs_K = K;
    /* child order of each emitted node (row of its node index), K entries */
    int32_t* ord = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B + 1) * K);
    int32_t* crank = (int32_t*)calloc((size_t)B + 1, sizeof(int32_t)); /* candidate rank per node */
    or_heap h = { 0, 0, 0 };
    if (!ord || !crank) { free(ord); free(crank); return OR_ENOMEM; }
    crank[0] = 0; /* the root's edge row */
    or_hs_order(1, 0, K, ord);
    or_node first;
    memset(&first, 0, sizeof first);
    first.d = 1; first.r[0] = 0; first.parent = 0;
    first.s = 0.0f + or_hs_edge(1, 0, ord[0]);
    int rc = or_heap_push(&h, &first);
    int n = 0;
    while (rc == OR_OK && n < B && h.n > 0) {
        or_node x = or_heap_pop(&h);
        int p = x.parent, jpos = x.r[x.d - 1];
        int c = ord[(size_t)p * K + jpos]; /* candidate rank at position x.d */
        ++n;
        if (n >= Mmax) { rc = OR_EINVAL; break; }
        tok[n] = id[(x.d - 1) * K + c];
        parent[n] = p;
        depth[n] = x.d;
        rank[n] = c;
        score[n] = x.s;
        crank[n] = c;
        if (x.d < L) {
            or_hs_order(x.d + 1, c, K, ord + (size_t)n * K);
            or_node ch = x;
            ch.d = x.d + 1; ch.r[x.d] = 0; ch.parent = n;
            ch.s = x.s + or_hs_edge(ch.d, c, ord[(size_t)n * K]);
            rc = or_heap_push(&h, &ch);
        }
        if (rc == OR_OK && jpos + 1 < K) {
            or_node sib = x;
            sib.r[x.d - 1] = jpos + 1;
            sib.s = score[p] + or_hs_edge(x.d, crank[p], ord[(size_t)p * K + jpos + 1]);
            rc = or_heap_push(&h, &sib);
        }
    }
    *n_nodes = n + 1;
    free(ord); free(crank); free(h.a);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* TALON budgeted, confidence-gated expansion.                                 */
/* [TALON] "Key designs" 1 (root layer keeps the Top-k children regardless of  */
/* confidence, k = 10 by default) and 2 (pool = children of every node of the  */
/* last layer, path probability p(u) = p(v) * P(w | x<=v), anchor m_d = max   */
/* p(u) over the pool, keep p(u) >= mu * m_d; when the layer passing the gate  */
/* exceeds the remaining budget N - |T|, keep its best N - |T| nodes and       */
/* stop).                                                                      */
/* Log domain: s(u) = s(v) + lp_d(w) in fp32; gate s(u) >= m_d + log_mu with   */
/* log_mu = log(mu) rounded to fp32 by the caller.  For a block drafter        */
/* P(w | x<=v) is the marginal at that position, so lp_d comes from the        */
/* position's candidate list.  |T| excludes the root.  The list may be the     */
/* full vocabulary (Kc = V) or the top min(N, V); both give the same tree.     */
/* Pinned: hand-computed V=4 case (golden), invariants, full-list equality.    */
/* ------------------------------------------------------------------------- */
int or_talon(const float* lp, const int32_t* id, int L, int Kc, int talon_k,
             float log_mu, int N, int Mmax,
             int32_t* tok, int32_t* parent, int32_t* depth, int32_t* rank,
             float* score, int32_t* n_nodes)
{
    if (L < 1 || L > OR_MAXL || Kc < 1 || talon_k < 1 || N < 1 || Mmax < N + 1) return OR_EINVAL;
    or_node* T = (or_node*)calloc((size_t)N + 1, sizeof(or_node));
    if (!T) return OR_ENOMEM;
    int nT = 0;
    int k1 = talon_k;
    if (k1 > Kc) k1 = Kc;
    if (k1 > N) k1 = N;
    for (int r = 0; r < k1; ++r) {
        or_node* x = &T[nT];
        x->d = 1; x->r[0] = r; x->s = lp[r]; x->tok = id[r]; x->parent = -1;
        x->self = nT;
        ++nT;
    }
    int lay_lo = 0, lay_hi = nT;
    or_node* pool = NULL;
    int rc = OR_OK;
    for (int d = 2; d <= L && nT < N; ++d) {
        int np = (lay_hi - lay_lo) * Kc;
        or_node* np_pool = (or_node*)realloc(pool, (size_t)np * sizeof(or_node));
        if (!np_pool) { rc = OR_ENOMEM; break; }
        pool = np_pool;
        int k = 0;
        float m_d = -INFINITY;
        for (int v = lay_lo; v < lay_hi; ++v)
            for (int w = 0; w < Kc; ++w) {
                or_node* x = &pool[k++];
                *x = T[v];
                x->d = d;
                x->r[d - 1] = w;
                x->s = T[v].s + lp[(d - 1) * Kc + w];
                x->tok = id[(d - 1) * Kc + w];
                x->parent = v;
                if (x->s > m_d) m_d = x->s;
            }
        float thr = m_d + log_mu;
        int npass = 0;
        for (int i = 0; i < k; ++i)
            if (pool[i].s >= thr) pool[npass++] = pool[i];
        int room = N - nT;
        int stop = 0;
        if (npass > room) {
            qsort(pool, (size_t)npass, sizeof(or_node), or_cmp_node);
            npass = room;
            stop = 1;
        }
        lay_lo = nT;
        for (int i = 0; i < npass; ++i) { T[nT] = pool[i]; T[nT].self = nT; ++nT; }
        lay_hi = nT;
        if (stop || npass == 0) break;
    }
    free(pool);
    if (rc != OR_OK) { free(T); return rc; }
    /* output: root, then T by the shared node order */
    or_node* srt = (or_node*)malloc((size_t)nT * sizeof(or_node));
    memcpy(srt, T, (size_t)nT * sizeof(or_node));
    qsort(srt, (size_t)nT, sizeof(or_node), or_cmp_node);
    int* out_of = (int*)malloc((size_t)(nT > 0 ? nT : 1) * sizeof(int));
    for (int i = 0; i < nT; ++i) out_of[srt[i].self] = i + 1;
    or_tree_out o = { tok, parent, depth, rank, score };
    or_put_root(&o);
    for (int i = 0; i < nT; ++i) {
        const or_node* x = &srt[i];
        tok[i + 1] = x->tok;
        parent[i + 1] = x->parent < 0 ? 0 : out_of[x->parent];
        depth[i + 1] = x->d;
        rank[i + 1] = x->r[x->d - 1];
        score[i + 1] = x->s;
    }
    *n_nodes = nT + 1;
    free(srt); free(out_of); free(T);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Tree-attention mask and position ids.                                       */
/* [DARTree] "Tree verification and DDTree" (each flattened node attends to    */
/* the verified context and the tokens on its root-to-node path); [DDTree]     */
/* section 4.2 (parent's global index per token, mask by path).                */
/* mask[n][m] = 1 iff m is an ancestor of n or n itself, bit m%32 of word m/32 */
/* of row n; row stride ceil(Mmax/32) words; pos[n] = depth(n) + pos_offset.   */
/* Validation: parent[0] = -1, depth[0] = 0, and for n >= 1 the parent lies in */
/* [0, M), differs from n, and depth(n) = depth(parent) + 1.                   */
/* Pinned: hand-drawn depth-3 tree (golden), popcount and closure invariants.  */
/* ------------------------------------------------------------------------- */
static int or_tree_valid(const int32_t* parent, const int32_t* depth, int M, int L)
{
    if (M < 1) return 0;
    if (parent[0] != -1 || depth[0] != 0) return 0;
    for (int n = 1; n < M; ++n) {
        int p = parent[n];
        if (p < 0 || p >= M || p == n) return 0;
        if (depth[n] != depth[p] + 1) return 0;
        if (L > 0 && depth[n] > L) return 0;
    }
    return 1;
}

int or_tree_mask(const int32_t* parent, const int32_t* depth, int M, int Mmax,
                 int L, int pos_offset, uint32_t* mask, int32_t* pos)
{
    if (M > Mmax) return OR_EINVAL;
    if (!or_tree_valid(parent, depth, M, L)) return OR_EBADTREE;
    int words = (Mmax + 31) / 32;
    for (int n = 0; n < M; ++n) {
        uint32_t* row = mask + (int64_t)n * words;
        for (int w = 0; w < words; ++w) row[w] = 0u;
        for (int a = n; a != -1; a = parent[a]) row[a / 32] |= 1u << (a % 32);
        pos[n] = depth[n] + pos_offset;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Greedy (T=0) tree verification.                                             */
/* [DARTree] "Speculative sampling" (T=0 accepts draft tokens that match the   */
/* target's greedy choice; at the first mismatch the target's choice is        */
/* emitted); [Unit11] temperature section (greedy ties go to the smallest      */
/* vocabulary index); [Unit11] bonus-token section (when the walk reaches a    */
/* node with nothing left to verify, the target row of that node yields one    */
/* more token).                                                                */
/* Walk from the root: a = argmax of target row n; descend into the child of n */
/* whose token is a, if any; otherwise stop.  Emits a.                         */
/* acc_nodes[0] = 0 (root), acc_nodes[1..acc_len] the accepted nodes, the rest */
/* -1.  visited rows only.                                                     */
/* Pinned: chain tree = sequential greedy decoding; hash-defined target (the   */
/* accepted path equals greedy decoding until it leaves the tree); a tie of    */
/* two tokens goes to the smaller id (tests).                                  */
/* ------------------------------------------------------------------------- */
int or_verify_greedy(const int32_t* tok, const int32_t* parent, const int32_t* depth,
                     int M, int L, const float* target, int V,
                     int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok)
{
    if (!or_tree_valid(parent, depth, M, L)) return OR_EBADTREE;
    for (int i = 0; i <= L; ++i) acc_nodes[i] = -1;
    int n = 0, len = 0, a = -1;
    acc_nodes[0] = 0;
    for (;;) {
        const float* row = target + (int64_t)n * V;
        a = 0;
        for (int v = 1; v < V; ++v)
            if (row[v] > row[a]) a = v;
        int child = -1;
        for (int c = 1; c < M && child < 0; ++c)
            if (parent[c] == n && tok[c] == a) child = c;
        if (child < 0 || len >= L) break;
        acc_nodes[++len] = child;
        n = child;
    }
    *acc_len = len;
    *next_tok = a;
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Stochastic (T=1) tree verification.                                         */
/* [DARTree] "Speculative sampling" (accept y ~ q with min(1, p/q); on the     */
/* first rejection draw one replacement from the normalised residual           */
/* [p - q]_+); [Unit11] worked three-token example, probability tree and       */
/* histogram proofs (R = 0 skips the residual; p(x) = 0 < q(x) always         */
/* rejects); [Unit11] bonus-token section (a fully accepted path samples one   */
/* more token from the target row).                                            */
/* On a tree (the pages state the single-chain rule): at node n, test the      */
/* children of n in rank order; child c is accepted iff                        */
/*   u[0][c] < exp_canon((t_n[tok c] - lse_t) - (d_{pos c}[tok c] - lse_d)),   */
/* and the walk descends into the first accepted child.  If n has children and */
/* all are rejected, draw from w(v) = max(0, P(v) - Q(v)) with P, Q the        */
/* fixed-point masses floor(exp_canon(.) * 2^32) of the target row of n and of */
/* the drafter row of n's children's position; if that residual is empty draw  */
/* from P.  A node without children draws its bonus token from P.  The draw:   */
/* X = floor(u[1][n] * 2^24), target = floor(X * S / 2^24), emit the smallest  */
/* v whose inclusive prefix sum of weights exceeds target.                     */
/* lse_t of each visited row is computed here (double, rounded to fp32) unless */
/* lse_in supplies it per node ([Mmax], row n's normaliser); lse_out receives  */
/* the values used, per step of the walk.                                      */
/* Pinned: worked example through a one-child chain, output frequencies equal  */
/* p within 3 sigma, R = 0 and p = 0 edge cases, a uniform of exactly 1/2 over */
/* two equal masses draws the second token (tests).                            */
/* ------------------------------------------------------------------------- */
static uint64_t or_fixed32(float p)
{
    float f = p * 4294967296.0f;
    return (uint64_t)f;
}

static int or_draw(const uint64_t* w, int V, uint64_t S, float u)
{
    float xf = u * 16777216.0f;
    uint64_t X = (uint64_t)xf;
    if (X > 16777215u) X = 16777215u;
    unsigned __int128 prod = (unsigned __int128)X * (unsigned __int128)S;
    uint64_t target = (uint64_t)(prod >> 24);
    uint64_t acc = 0;
    int last = -1;
    for (int v = 0; v < V; ++v) {
        if (w[v] == 0) continue;
        acc += w[v];
        last = v;
        if (acc > target) return v;
    }
    return last;
}

static float or_row_lse(const float* row, int V)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) if ((double)row[v] > m) m = (double)row[v];
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp((double)row[v] - m);
    return (float)(m + log(s));
}

int or_verify_t1(const int32_t* tok, const int32_t* parent, const int32_t* depth,
                 const int32_t* rank, int M, int L, int Mmax,
                 const float* target, const float* draft, const float* draft_lse,
                 int V, const float* u, const float* lse_in,
                 int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                 float* lse_out)
{
    if (!or_tree_valid(parent, depth, M, L)) return OR_EBADTREE;
    uint64_t* w = (uint64_t*)malloc((size_t)V * sizeof(uint64_t));
    int* kids = (int*)malloc((size_t)M * sizeof(int));
    if (!w || !kids) { free(w); free(kids); return OR_ENOMEM; }
    for (int i = 0; i <= L; ++i) { acc_nodes[i] = -1; if (lse_out) lse_out[i] = 0.0f; }
    int n = 0, len = 0, out = -1;
    acc_nodes[0] = 0;
    for (;;) {
        const float* trow = target + (int64_t)n * V;
        float lse_t = lse_in ? lse_in[n] : or_row_lse(trow, V);
        if (lse_out) lse_out[len] = lse_t;
        /* children of n in rank order (insertion sort; ranks are distinct) */
        int nk = 0;
        for (int c = 1; c < M; ++c)
            if (parent[c] == n) {
                int j = nk++;
                while (j > 0 && rank[kids[j - 1]] > rank[c]) { kids[j] = kids[j - 1]; --j; }
                kids[j] = c;
            }
        int acc = -1;
        for (int i = 0; i < nk && acc < 0; ++i) {
            int c = kids[i];
            int pos = depth[c] - 1;
            float lpt = trow[tok[c]] - lse_t;
            float lpq = draft[(int64_t)pos * V + tok[c]] - draft_lse[pos];
            float ratio = or_exp_canon(lpt - lpq);
            if (u[c] < ratio) acc = c;
        }
        if (acc >= 0 && len < L) {
            acc_nodes[++len] = acc;
            n = acc;
            continue;
        }
        uint64_t S = 0;
        if (nk > 0) {
            int pos = depth[n];
            const float* drow = draft + (int64_t)pos * V;
            float lsed = draft_lse[pos];
            for (int v = 0; v < V; ++v) {
                uint64_t P = or_fixed32(or_exp_canon(trow[v] - lse_t));
                uint64_t Q = or_fixed32(or_exp_canon(drow[v] - lsed));
                w[v] = P > Q ? P - Q : 0;
                S += w[v];
            }
        }
        if (S == 0) {
            for (int v = 0; v < V; ++v) {
                w[v] = or_fixed32(or_exp_canon(trow[v] - lse_t));
                S += w[v];
            }
        }
        out = or_draw(w, V, S, u[Mmax + n]);
        break;
    }
    *acc_len = len;
    *next_tok = out;
    free(w); free(kids);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* T=1 tree verification against the normalised DARTree proposal.             */
/* [DARTree] "Causal correction" (with the full-vocabulary normaliser the       */
/* corrected distribution q~(. | u) is a probability, which is what lets the   */
/* speculative-sampling test of "Speculative sampling" use it): at node n, the */
/* drafter proposes n's children from                                          */
/*   log q~(v | u) = ((d_pos[v] - lse_pos) + <U[u], Vt[v]>) - z,               */
/* u = tok(n) (the root: root_tok), pos = depth(n) (the children's position),  */
/* z = znorm[pos][rank(n)] (the root: znorm[0][0]), each step rounded to fp32, */
/* the dot product the serial fmaf chain of or_markov.  Without a parent token */
/* (the root and root_tok < 0) q~ is the plain marginal.  Otherwise the rule   */
/* of or_verify_t1: children in rank order, u[0][c] < exp_canon(lpt - log q~), */
/* first acceptance descends, the replacement from max(0, P - Q~), Q~ the 2^32 */
/* fixed-point masses of q~, or from P when that is empty or n has no          */
/* children.                                                                   */
/* Pinned: U = 0 and z = 0 give or_verify_t1; the proposal sums to 1 with the  */
/* exact normaliser; a chain whose child is drawn from q~ emits p (tests).     */
/* ------------------------------------------------------------------------- */
int or_verify_t1_markov(const int32_t* tok, const int32_t* parent, const int32_t* depth,
                        const int32_t* rank, int M, int L, int Mmax,
                        const float* target, const float* draft, const float* draft_lse,
                        int V, const float* U, const float* Vt, int R, int root_tok,
                        const float* znorm /* [L][K] */, int K,
                        const float* u, const float* lse_in,
                        int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok)
{
    if (!or_tree_valid(parent, depth, M, L)) return OR_EBADTREE;
    if (!U || !Vt || R < 1 || !znorm || K < 1) return OR_EINVAL;
    uint64_t* w = (uint64_t*)malloc((size_t)V * sizeof(uint64_t));
    int* kids = (int*)malloc((size_t)M * sizeof(int));
    if (!w || !kids) { free(w); free(kids); return OR_ENOMEM; }
    for (int i = 0; i <= L; ++i) acc_nodes[i] = -1;
    int n = 0, len = 0, out = -1;
    acc_nodes[0] = 0;
    for (;;) {
        const float* trow = target + (int64_t)n * V;
        float lse_t = lse_in ? lse_in[n] : or_row_lse(trow, V);
        int ptok = n == 0 ? root_tok : tok[n];
        int pos = depth[n];
        float z = 0.0f;
        if (ptok >= 0 && pos < L) z = znorm[pos * K + (n == 0 ? 0 : rank[n])];
        int nk = 0;
        for (int c = 1; c < M; ++c)
            if (parent[c] == n) {
                int j = nk++;
                while (j > 0 && rank[kids[j - 1]] > rank[c]) { kids[j] = kids[j - 1]; --j; }
                kids[j] = c;
            }
        const float* drow = pos < L ? draft + (int64_t)pos * V : NULL;
        float lsed = pos < L ? draft_lse[pos] : 0.0f;
        int acc = -1;
        for (int i = 0; i < nk && acc < 0; ++i) {
            int c = kids[i];
            float lpt = trow[tok[c]] - lse_t;
            float lpq = drow[tok[c]] - lsed;
            if (ptok >= 0) { lpq = lpq + or_markov(U, Vt, R, ptok, tok[c]); lpq = lpq - z; }
            if (u[c] < or_exp_canon(lpt - lpq)) acc = c;
        }
        if (acc >= 0 && len < L) {
            acc_nodes[++len] = acc;
            n = acc;
            continue;
        }
        uint64_t S = 0;
        if (nk > 0) {
            for (int v = 0; v < V; ++v) {
                float lpq = drow[v] - lsed;
                if (ptok >= 0) { lpq = lpq + or_markov(U, Vt, R, ptok, v); lpq = lpq - z; }
                uint64_t P = or_fixed32(or_exp_canon(trow[v] - lse_t));
                uint64_t Q = or_fixed32(or_exp_canon(lpq));
                w[v] = P > Q ? P - Q : 0;
                S += w[v];
            }
        }
        if (S == 0) {
            for (int v = 0; v < V; ++v) {
                w[v] = or_fixed32(or_exp_canon(trow[v] - lse_t));
                S += w[v];
            }
        }
        out = or_draw(w, V, S, u[Mmax + n]);
        break;
    }
    *acc_len = len;
    *next_tok = out;
    free(w); free(kids);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Tree verification at T=1 with one residual per rejected sibling.            */
/* [Unit11] residual formula: after drafting y ~ q is rejected, the output is   */
/* drawn from r = [p - q]_+ / sum [p - q]_+; [DARTree] "Speculative sampling"  */
/* (the same rule).  The pages state it for one drafted token per position;    */
/* with several children at a node the plain extension applies it once per     */
/* rejected child: child c_1 is tested against p, child c_i (i >= 2) against   */
/* the residual r_{i-1} left by the rejections of c_1 .. c_{i-1}, where         */
/*   r_0 = p,   r_i = [r_{i-1} - q]_+ / sum [r_{i-1} - q]_+,                    */
/* and the replacement is drawn from r_k after all k children are rejected.    */
/* Exact integer form: with P, Q the 2^32 fixed-point masses (as in            */
/* or_verify_t1), r_i is proportional to                                       */
/*   W_i(v) = max(0, P(v) - floor(Q(v) * T_i / 2^32)),                          */
/*   T_1 = 2^32 (the nominal mass of P),  T_{i+1} = T_i + S_i,  S_i = sum W_i,  */
/* since subtracting S_i * q from [P - T_i q]_+ and clamping at zero equals     */
/* [P - (T_i + S_i) q]_+.  Child c_1 takes or_verify_t1's test; child c_i       */
/* (i >= 2) is accepted iff floor(u * 2^24) * Q(c) * S_{i-1}                    */
/*   < W_{i-1}(c) * 2^56, i.e. u < r_{i-1}(c) / q(c) in exact integers.         */
/* When a residual is empty (S_i = 0) the remaining children are not tested    */
/* and the draw is from P, as in or_verify_t1.  With one child per node this   */
/* is or_verify_t1 exactly.  The draw uses or_draw with uniforms[1][n].        */
/* Pinned: equals or_verify_t1 on single-child trees; with the children's      */
/* tokens drawn i.i.d. from q the emitted first token follows p (frequency     */
/* test), the losslessness of the iterated rule for sampled candidates (tests). */
/* ------------------------------------------------------------------------- */
static uint64_t or_qscale(uint64_t Q, uint64_t T)
{
    return (uint64_t)(((unsigned __int128)Q * (unsigned __int128)T) >> 32);
}

static uint64_t or_resid_w(uint64_t P, uint64_t Q, uint64_t T)
{
    uint64_t s = or_qscale(Q, T);
    return P > s ? P - s : 0;
}

static int or_accept_resid(float u, uint64_t Q, uint64_t S, uint64_t W)
{
    float xf = u * 16777216.0f;
    uint64_t X = (uint64_t)xf;
    if (X > 16777215u) X = 16777215u;
    unsigned __int128 lhs = (unsigned __int128)(X * Q) * (unsigned __int128)S;
    unsigned __int128 rhs = (unsigned __int128)W << 56;
    return lhs < rhs;
}

int or_verify_iter_residual(const int32_t* tok, const int32_t* parent, const int32_t* depth,
                            const int32_t* rank, int M, int L, int Mmax,
                            const float* target, const float* draft, const float* draft_lse,
                            int V, const float* u, const float* lse_in,
                            int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                            float* lse_out)
{
    if (!or_tree_valid(parent, depth, M, L)) return OR_EBADTREE;
    uint64_t* w = (uint64_t*)malloc((size_t)V * sizeof(uint64_t));
    uint64_t* P = (uint64_t*)malloc((size_t)V * sizeof(uint64_t));
    uint64_t* Q = (uint64_t*)malloc((size_t)V * sizeof(uint64_t));
    int* kids = (int*)malloc((size_t)M * sizeof(int));
    if (!w || !P || !Q || !kids) { free(w); free(P); free(Q); free(kids); return OR_ENOMEM; }
    for (int i = 0; i <= L; ++i) { acc_nodes[i] = -1; if (lse_out) lse_out[i] = 0.0f; }
    int n = 0, len = 0, out = -1;
    acc_nodes[0] = 0;
    for (;;) {
        const float* trow = target + (int64_t)n * V;
        float lse_t = lse_in ? lse_in[n] : or_row_lse(trow, V);
        if (lse_out) lse_out[len] = lse_t;
        int nk = 0;
        for (int c = 1; c < M; ++c)
            if (parent[c] == n) {
                int j = nk++;
                while (j > 0 && rank[kids[j - 1]] > rank[c]) { kids[j] = kids[j - 1]; --j; }
                kids[j] = c;
            }
        int acc = -1;
        uint64_t S = 0;
        if (nk > 0) {
            int pos = depth[n]; /* the children's position */
            const float* drow = draft + (int64_t)pos * V;
            float lsed = draft_lse[pos];
            for (int v = 0; v < V; ++v) {
                P[v] = or_fixed32(or_exp_canon(trow[v] - lse_t));
                Q[v] = or_fixed32(or_exp_canon(drow[v] - lsed));
            }
            /* c_1 against p */
            int c = kids[0];
            float lpt = trow[tok[c]] - lse_t;
            float lpq = drow[tok[c]] - lsed;
            if (u[c] < or_exp_canon(lpt - lpq)) acc = c;
            /* c_2 .. c_k against the residuals */
            uint64_t T = (uint64_t)1 << 32;
            for (int i = 1; acc < 0; ++i) {
                S = 0;
                for (int v = 0; v < V; ++v) { w[v] = or_resid_w(P[v], Q[v], T); S += w[v]; }
                if (i == nk || S == 0) break;
                c = kids[i];
                if (or_accept_resid(u[c], Q[tok[c]], S, w[tok[c]])) acc = c;
                else T += S;
            }
        }
        if (acc >= 0 && len < L) {
            acc_nodes[++len] = acc;
            n = acc;
            continue;
        }
        if (S == 0) {
            for (int v = 0; v < V; ++v) {
                w[v] = or_fixed32(or_exp_canon(trow[v] - lse_t));
                S += w[v];
            }
        }
        out = or_draw(w, V, S, u[Mmax + n]);
        break;
    }
    *acc_len = len;
    *next_tok = out;
    free(w); free(P); free(Q); free(kids);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Tree verification at T=1 by exact target-sample matching.                   */
/* [DARTree] "Speculative sampling": some systems (DFlash) do not run the       */
/* rejection procedure and instead match a sample of the target against the    */
/* draft.  On a tree: at node n draw y from the target row of n (P, the 2^32    */
/* fixed-point masses, or_draw with uniforms[1][n]); if a child of n carries    */
/* token y, accept it and continue from it; otherwise emit y.  A node without   */
/* children emits its draw as the bonus token.  Every emitted token is a       */
/* target sample given the accepted prefix, so the output follows the target   */
/* distribution whatever the tree.  The drafter rows are not used.              */
/* Pinned: the emitted first token follows p (frequency test); with one-hot     */
/* target rows it is the greedy walk (tests).                                   */
/* ------------------------------------------------------------------------- */
int or_verify_target_match(const int32_t* tok, const int32_t* parent, const int32_t* depth,
                           int M, int L, int Mmax, const float* target, int V,
                           const float* u, const float* lse_in,
                           int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                           float* lse_out)
{
    if (!or_tree_valid(parent, depth, M, L)) return OR_EBADTREE;
    uint64_t* w = (uint64_t*)malloc((size_t)V * sizeof(uint64_t));
    if (!w) return OR_ENOMEM;
    for (int i = 0; i <= L; ++i) { acc_nodes[i] = -1; if (lse_out) lse_out[i] = 0.0f; }
    int n = 0, len = 0, y = -1;
    acc_nodes[0] = 0;
    for (;;) {
        const float* trow = target + (int64_t)n * V;
        float lse_t = lse_in ? lse_in[n] : or_row_lse(trow, V);
        if (lse_out) lse_out[len] = lse_t;
        uint64_t S = 0;
        for (int v = 0; v < V; ++v) {
            w[v] = or_fixed32(or_exp_canon(trow[v] - lse_t));
            S += w[v];
        }
        y = or_draw(w, V, S, u[Mmax + n]);
        int child = -1;
        for (int c = 1; c < M && child < 0; ++c)
            if (parent[c] == n && tok[c] == y) child = c;
        if (child < 0 || len >= L) break;
        acc_nodes[++len] = child;
        n = child;
    }
    *acc_len = len;
    *next_tok = y;
    free(w);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Single-position speculative sampling in double precision, the scalar rule   */
/* the tree walk generalises.  [Unit11] worked three-token example and its     */
/* probability-tree / histogram proofs; [DARTree] "Speculative sampling".      */
/* Draw x ~ q by inverse CDF from u_draw; accept with a = min(1, p(x)/q(x))    */
/* (a = 1 when q(x) = 0 is never needed: x ~ q has q(x) > 0); on rejection     */
/* draw from r = (p - q)_+ / R by inverse CDF from u_res.  Outputs the accept  */
/* probability of each token and the residual distribution (zeros if R = 0).  */
/* Pinned: worked example values (golden), frequency test (tests).             */
/* ------------------------------------------------------------------------- */
int or_spec_scalar(const double* p, const double* q, int n, double u_draw,
                   double u_acc, double u_res, double* accept_prob,
                   double* residual, int32_t* drafted)
{
    double R = 0.0;
    for (int i = 0; i < n; ++i) {
        accept_prob[i] = q[i] > 0.0 ? (p[i] < q[i] ? p[i] / q[i] : 1.0) : 1.0;
        double z = p[i] - q[i];
        residual[i] = z > 0.0 ? z : 0.0;
        R += residual[i];
    }
    for (int i = 0; i < n; ++i) residual[i] = R > 0.0 ? residual[i] / R : 0.0;
    int x = n - 1;
    double c = 0.0;
    for (int i = 0; i < n; ++i) { c += q[i]; if (u_draw < c) { x = i; break; } }
    if (drafted) *drafted = x;
    if (u_acc < accept_prob[x]) return x;
    if (R <= 0.0) return x; /* unreachable: R = 0 means p = q and a = 1 */
    int y = n - 1;
    c = 0.0;
    for (int i = 0; i < n; ++i) { c += residual[i]; if (u_res < c) { y = i; break; } }
    return y;
}

/* Many trials of or_spec_scalar from a caller-supplied stream of uniforms
 * (three per trial), counting how often each token is emitted. */
int or_spec_scalar_trials(const double* p, const double* q, int n,
                          const double* uniforms, int64_t trials, int64_t* counts)
{
    double* a = (double*)malloc((size_t)n * sizeof(double));
    double* r = (double*)malloc((size_t)n * sizeof(double));
    if (!a || !r) { free(a); free(r); return OR_ENOMEM; }
    for (int i = 0; i < n; ++i) counts[i] = 0;
    for (int64_t t = 0; t < trials; ++t) {
        int y = or_spec_scalar(p, q, n, uniforms[3 * t], uniforms[3 * t + 1],
                               uniforms[3 * t + 2], a, r, NULL);
        counts[y] += 1;
    }
    free(a); free(r);
    return OR_OK;
}
