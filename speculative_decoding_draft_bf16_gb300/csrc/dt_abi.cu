// dt_abi.cu -- the library's C ABI: argument checks, launch shapes, and the
// entry points declared in include/dtree.h.
#include <cuda_runtime.h>

#include <mutex>

#include "dt_launch.h"
#include "dtree.h"

namespace {

constexpr int kChunkMax = 32768;       // vocabulary elements per CTA (shared memory)
constexpr int kCtaTarget = 2 * 152;    // aim for two CTAs per SM on a GB300
constexpr size_t kSmemMax = 227 * 1024;

int pow2_ceil(long long n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

int chunk_of(int V, int S, int dtype) {
    const int g = dtype == DT_BF16 ? 8 : 4;  // elements per 16 bytes
    long long per = ((long long)V + S - 1) / S;
    return (int)(((per + g - 1) / g) * g);
}

// Clusters of S CTAs that the device holds at once for stage 1 (kind 1,
// extra = Kc) or the verification walk (kind 6, extra = 8 * max_nodes + rule)
// with these sizes; cached per device.
int max_clusters(int kind, int dtype, int S, int chunk, int extra) {
    struct Fit {
        int dev, kind, dtype, S, chunk, extra, n;
    };
    static std::mutex mu;
    static Fit fits[128];
    static int nfit = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < nfit; ++i) {
        const Fit& f = fits[i];
        if (f.dev == dev && f.kind == kind && f.dtype == dtype && f.S == S && f.chunk == chunk && f.extra == extra)
            return f.n;
    }
    const int n = kind == 1 ? dt_kn1_max_clusters(dtype, S, chunk, extra)
                            : dt_kn6_max_clusters(dtype, S, chunk, extra >> 3, extra & 7);
    if (n > 0 && nfit < 128) fits[nfit++] = Fit{dev, kind, dtype, S, chunk, extra, n};
    return n;
}

// Stage 1 gives each row a CTA of its own (kn1b_rows.cu) instead of spreading
// it over a cluster (kn1_candidates.cu) from this many rows on, or for
// candidate lists longer than kRowsPerCtaKc at any row count (measured on a
// GB300 at V = 151936: both take ~21-25 us at 64 rows; at 16 rows the cluster
// kernel is faster for Kc <= 256, the row kernel for Kc = 1024).
#ifndef DT_KN1B_MIN_ROWS
#define DT_KN1B_MIN_ROWS 64
#endif
constexpr long long kRowsPerCtaMin = DT_KN1B_MIN_ROWS;
constexpr int kRowsPerCtaKc = 512;

// Per-CTA cost of a row pass that does not scale with its chunk (staging
// latency, cluster barriers, exchanges), in element-equivalents.
constexpr long long kFixedElems = 12288;

// Cluster size for a row-parallel vocabulary pass over `rows` rows (one
// cluster per row): the size in [s_min, 16] -- a power of two unless any_size
// -- with chunks of at most kChunkMax elements, and of at least ~1K unless that
// is s_min, that minimises the estimated time, waves x (chunk + kFixedElems),
// where a wave is as many clusters as the device holds at once.  smem_ok(S)
// says whether a cluster size fits in shared memory; fits(S) gives the
// resident clusters.  (Clusters are placed within a GPC, so how many fit
// depends on the size in ways only the occupancy query knows: on a GB300 at
// one CTA per SM, 15 clusters of 8 but more of 7.)
template <typename SmemOk, typename Fits>
int cluster_for(int V, long long rows, int dtype, SmemOk smem_ok, Fits fits, bool any_size = false) {
    // any size: the kernel has an SM to itself, so only its shared memory
    // (smem_ok) bounds the chunk; powers of two: chunks of at most kChunkMax
    int s_min = any_size ? (int)(((long long)V + 65535) / 65536)
                         : pow2_ceil(((long long)V + kChunkMax - 1) / kChunkMax);
    int s_cap = pow2_ceil(((long long)V + 1023) / 1024);  // chunks of at least ~1K elements
    if (s_cap > 16) s_cap = 16;
    if (s_min < 1) s_min = 1;
    if (s_cap < s_min) s_cap = s_min;
    int best = s_min;
    long long best_cost = -1;
    for (int s = s_min; s <= s_cap; s = any_size ? s + 1 : s << 1) {
        if (!smem_ok(s)) continue;
        const int chunk = chunk_of(V, s, dtype);
        int n = fits(s, chunk);
        if (n < 1) n = (int)((kCtaTarget + s - 1) / s);  // unknown: assume two CTAs per SM
        const long long waves = (rows + n - 1) / n;
        const long long cost = waves * (chunk + kFixedElems);
        if (best_cost < 0 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

dt_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DT_OK;
    (void)cudaGetLastError();
    return DT_ERR_CUDA;
}

int kc_of(const dt_build_params* p) {
    if (p->mode == DT_MODE_TALON) return p->N < p->V ? p->N : p->V;
    return p->K;
}

int budget_of(const dt_build_params* p) { return p->mode == DT_MODE_TALON ? p->N : p->B; }

// The Markov term <U, Vt> is on: DARTree, or the heap without a TDES scorer.
bool markov_on(const dt_build_params* p) {
    return (p->mode == DT_MODE_DARTREE || (p->mode == DT_MODE_HEAP && !p->tdes)) && p->R > 0 && p->U;
}

// DARTree layer width: W, or the largest per-depth width of the uniform budget.
int dartree_w(const dt_build_params* p) {
    return p->budget_policy == DT_BUDGET_UNIFORM ? (p->B + p->L - 1) / p->L : p->W;
}

// A per-request edge table lives in the workspace.
bool table_on(const dt_build_params* p) { return markov_on(p) || (p->mode == DT_MODE_HEAP && p->tdes); }

dt_status check_build(const dt_build_params* p, const dt_tree* t) {
    if (!p || !t) return DT_ERR_INVALID_ARG;
    if (p->mode < DT_MODE_DDTREE || p->mode > DT_MODE_HEAP) return DT_ERR_INVALID_ARG;
    if (p->batch < 1 || p->L < 1 || p->L > DT_MAX_L || p->V < 1) return DT_ERR_INVALID_ARG;
    if (p->V > DT_MAX_V) return DT_ERR_UNSUPPORTED;
    if (p->dtype != DT_BF16 && p->dtype != DT_F32) return DT_ERR_INVALID_ARG;
    if ((long long)p->batch * p->L > 65535) return DT_ERR_UNSUPPORTED;
    if (p->mode == DT_MODE_TALON) {
        if (p->N < 1 || p->N > DT_MAX_KC) return DT_ERR_INVALID_ARG;
        if (p->talon_k < 1 || p->talon_k > p->N) return DT_ERR_INVALID_ARG;
        if (!(p->log_mu <= 0.f) || p->log_mu != p->log_mu || p->log_mu == -__builtin_inff())
            return DT_ERR_INVALID_ARG;
    } else {
        if (p->K < 1 || p->K > p->V || p->K > DT_MAX_KC) return DT_ERR_INVALID_ARG;
        if (p->B < 1 || p->B > DT_MAX_NODES - 1) return DT_ERR_INVALID_ARG;
    }
    if (p->budget_policy != DT_BUDGET_TOPB && p->budget_policy != DT_BUDGET_UNIFORM) return DT_ERR_INVALID_ARG;
    if (p->budget_policy == DT_BUDGET_UNIFORM && (p->mode != DT_MODE_DARTREE || p->B < p->L)) return DT_ERR_INVALID_ARG;
    if (p->budget && p->mode != DT_MODE_DDTREE && p->mode != DT_MODE_HEAP) return DT_ERR_INVALID_ARG;
    if (p->mode == DT_MODE_DARTREE) {
        const int W = dartree_w(p);
        if (W < 1 || (long long)W * p->K > 4096 || (long long)W * p->L > 4096) return DT_ERR_INVALID_ARG;
        if (!(p->beta <= 0.f)) return DT_ERR_INVALID_ARG;  // Lemma 1 needs beta <= 0
        if (p->R < 0 || p->R > 1024) return DT_ERR_INVALID_ARG;
        if (p->R > 0 && (!p->U || !p->Vt)) return DT_ERR_INVALID_ARG;
        if (p->R > 0 && dt_kn3_table_smem_bytes(p->K, p->R) > kSmemMax) return DT_ERR_UNSUPPORTED;
        if (p->markov_norm != 0 && p->markov_norm != 1) return DT_ERR_INVALID_ARG;
        if (p->markov_norm && (p->R == 0 || !p->U)) return DT_ERR_INVALID_ARG;  // nothing to normalise
        if (p->markov_norm && p->R != 64) return DT_ERR_UNSUPPORTED;           // tensor-core tile: R = 64
        if (p->markov_norm && ((((uintptr_t)p->U) | ((uintptr_t)p->Vt)) & 15u)) return DT_ERR_INVALID_ARG;
        if (dt_kn3_select_smem_bytes(p->L, p->K, W, p->R > 0 && p->U) > kSmemMax) return DT_ERR_UNSUPPORTED;
    }
    if (p->mode == DT_MODE_HEAP) {
        if (p->K > 256) return DT_ERR_UNSUPPORTED;
        if (p->markov_norm != 0 && p->markov_norm != 1) return DT_ERR_INVALID_ARG;
        if (p->tdes) {
            const dt_tdes* q = p->tdes;
            if (q->H < 1 || q->H > 4096 || !q->Ap || !q->Ac || !q->Dd || !q->w) return DT_ERR_INVALID_ARG;
            if (p->markov_norm) return DT_ERR_INVALID_ARG;  // the normaliser is the Markov term's
            if (dt_kn8_smem_bytes(p->K, q->H) > kSmemMax) return DT_ERR_UNSUPPORTED;
        } else {
            if (p->R < 0 || p->R > 1024) return DT_ERR_INVALID_ARG;
            if (p->R > 0 && (!p->U || !p->Vt)) return DT_ERR_INVALID_ARG;
            if (p->R > 0 && dt_kn3_table_smem_bytes(p->K, p->R) > kSmemMax) return DT_ERR_UNSUPPORTED;
            if (p->markov_norm && (p->R == 0 || !p->U)) return DT_ERR_INVALID_ARG;
            if (p->markov_norm && p->R != 64) return DT_ERR_UNSUPPORTED;
            if (p->markov_norm && ((((uintptr_t)p->U) | ((uintptr_t)p->Vt)) & 15u)) return DT_ERR_INVALID_ARG;
        }
    }
    if (t->Kc != kc_of(p)) return DT_ERR_INVALID_ARG;
    if (t->L != p->L) return DT_ERR_INVALID_ARG;
    if (t->max_nodes < budget_of(p) + 1 || t->max_nodes > DT_MAX_NODES) {
        // DARTree needs room for min(B, |S|) nodes; DDTree and TALON for their budget
        if (!(p->mode == DT_MODE_DARTREE &&
              t->max_nodes >= 1 + ((p->B < dartree_w(p) * p->L) ? p->B : dartree_w(p) * p->L) &&
              t->max_nodes <= DT_MAX_NODES))
            return DT_ERR_INVALID_ARG;
    }
    if (!t->node_tok || !t->parent || !t->depth || !t->rank || !t->score || !t->n_nodes || !t->lse ||
        !t->cand_id || !t->cand_lp || !t->status)
        return DT_ERR_INVALID_ARG;
    return DT_OK;
}

// Bytes of the DARTree log-normaliser table (rounded up to 256).
size_t znorm_bytes(const dt_build_params* p) { return (((size_t)p->batch * p->L * p->K * 4) + 255) & ~(size_t)255; }

// Stage-1 launch shape: kernel DT_STAGE1_ROWS (one CTA per row) or
// DT_STAGE1_CLUSTER (a cluster of S CTAs, chunk elements each, per row).
struct Stage1Plan {
    int kernel, S, chunk;
};

dt_status plan_stage1(const dt_build_params* p, Stage1Plan* plan) {
    const int Kc = kc_of(p);
    const long long rows = (long long)p->batch * p->L;
    const int esize = p->dtype == DT_BF16 ? 2 : 4;
    const int V = p->V, dtype = p->dtype;
    // enough rows to fill the GPU with whole rows, or long candidate lists:
    // one CTA per row, no cluster
    if (rows >= kRowsPerCtaMin || Kc > kRowsPerCtaKc) {
        *plan = Stage1Plan{DT_STAGE1_ROWS, 1, V};
        return DT_OK;
    }
    const int S = cluster_for(
        V, rows, dtype, [&](int q) { return dt_kn1_smem_bytes(chunk_of(V, q, dtype), Kc, esize) + 4096 <= kSmemMax; },
        [&](int q, int chunk) { return max_clusters(1, dtype, q, chunk, Kc); }, true);
    const int chunk = chunk_of(V, S, dtype);
    if (dt_kn1_smem_bytes(chunk, Kc, esize) + 4096 > kSmemMax) return DT_ERR_UNSUPPORTED;
    *plan = Stage1Plan{DT_STAGE1_CLUSTER, S, chunk};
    return DT_OK;
}

}  // namespace

extern "C" {

size_t dt_workspace_size(const dt_build_params* p, int* ok) {
    if (ok) *ok = 1;
    if (!p || p->batch < 1 || p->L < 1 || p->K < 0) {
        if (ok) *ok = 0;
        return 0;
    }
    if (table_on(p)) {
        size_t n = DT_ZNORM_OFFSET(p);
        if (markov_on(p) && p->markov_norm)
            n += znorm_bytes(p) + dt_kn3n_scratch_bytes(p->batch * p->L * p->K, p->V);
        return n;
    }
    return 0;
}

dt_status dt_stage1_plan(const dt_build_params* p, int32_t* kernel, int32_t* cluster) {
    if (!p || !kernel || !cluster) return DT_ERR_INVALID_ARG;
    if (p->batch < 1 || p->L < 1 || p->L > DT_MAX_L || p->V < 1 || p->V > DT_MAX_V) return DT_ERR_INVALID_ARG;
    if (p->dtype != DT_BF16 && p->dtype != DT_F32) return DT_ERR_INVALID_ARG;
    const int Kc = kc_of(p);
    if (Kc < 1 || Kc > DT_MAX_KC || Kc > p->V) return DT_ERR_INVALID_ARG;
    Stage1Plan plan;
    const dt_status s = plan_stage1(p, &plan);
    if (s != DT_OK) return s;
    *kernel = plan.kernel;
    *cluster = plan.S;
    return DT_OK;
}

dt_status dt_stage1_ceiling(const dt_build_params* p, const void* draft_logits, float* chunk_max, int32_t* status,
                            dt_stream_t stream) {
    int32_t kernel = 0, S = 0;
    dt_status s = dt_stage1_plan(p, &kernel, &S);
    if (s != DT_OK) return s;
    if (!draft_logits || !chunk_max) return DT_ERR_INVALID_ARG;
    if (kernel != DT_STAGE1_CLUSTER) return DT_ERR_UNSUPPORTED;
    Stage1Plan plan;
    if ((s = plan_stage1(p, &plan)) != DT_OK) return s;
    return cuda_status(dt_kn0_launch(draft_logits, p->dtype, p->batch * p->L, p->V, kc_of(p), plan.S, plan.chunk,
                                     chunk_max, status, (cudaStream_t)stream));
}

dt_status dt_candidates(const dt_build_params* p, const void* draft_logits, dt_tree* t, dt_stream_t stream) {
    dt_status s = check_build(p, t);
    if (s != DT_OK) return s;
    if (!draft_logits) return DT_ERR_INVALID_ARG;
    Stage1Plan plan;
    if ((s = plan_stage1(p, &plan)) != DT_OK) return s;
    const int rows = p->batch * p->L;
    cudaError_t e;
    if (plan.kernel == DT_STAGE1_ROWS)
        e = dt_kn1b_launch(draft_logits, p->dtype, rows, p->V, kc_of(p), t->lse, t->cand_id, t->cand_lp,
                           (cudaStream_t)stream);
    else
        e = dt_kn1_launch(draft_logits, p->dtype, rows, rows, p->V, kc_of(p), plan.S, plan.chunk, t->lse,
                          t->cand_id, t->cand_lp, (cudaStream_t)stream);
    return cuda_status(e);
}

// Selection kernels, optionally also writing the tree mask and positions.
static dt_status select_impl(const dt_build_params* p, dt_tree* t, void* workspace, size_t workspace_bytes,
                             uint32_t* mask_out, int32_t* pos_out, int pos_offset, cudaStream_t st) {
    dt_status s = check_build(p, t);
    if (s != DT_OK) return s;
    cudaError_t e = cudaSuccess;
    const int Mmax = t->max_nodes;
    // The DDTree, DARTree and TALON kernels write the mask rows themselves,
    // walking parents in shared memory (dt_mask.cuh); the heap selection is
    // followed by the level-by-level mask kernel.
    const bool fuse = mask_out && p->mode != DT_MODE_HEAP;
    uint32_t* mask = fuse ? mask_out : nullptr;
    int32_t* pos = fuse ? pos_out : nullptr;
    switch (p->mode) {
        case DT_MODE_DDTREE:
            if (dt_kn2_smem_bytes(p->L, p->K, p->B) > kSmemMax) return DT_ERR_UNSUPPORTED;
            e = dt_kn2_launch(p->batch, p->L, p->K, p->B, p->budget, Mmax, t->cand_lp, t->cand_id, t->lse, t->node_tok,
                              t->parent, t->depth, t->rank, t->score, t->n_nodes, t->status, mask, pos, pos_offset, st);
            break;
        case DT_MODE_DARTREE: {
            const size_t need = dt_workspace_size(p, nullptr);
            if (need > 0 && (!workspace || workspace_bytes < need)) return DT_ERR_INVALID_ARG;
            const bool term = p->R > 0 && p->U;
            const float* znorm =
                (term && p->markov_norm) ? (const float*)((const unsigned char*)workspace + DT_ZNORM_OFFSET(p)) : nullptr;
            e = dt_kn3_launch(p->batch, p->L, p->V, p->K, dartree_w(p), p->budget_policy == DT_BUDGET_UNIFORM, p->B,
                              p->beta, term ? p->R : 0, p->U, p->Vt, p->root_tok,
                              Mmax, t->cand_lp, t->cand_id, t->lse, term ? (float*)workspace : nullptr, znorm,
                              t->node_tok, t->parent, t->depth, t->rank, t->score, t->n_nodes, t->status, mask, pos,
                              pos_offset, st);
            break;
        }
        case DT_MODE_HEAP: {
            const size_t need = dt_workspace_size(p, nullptr);
            if (need > 0 && (!workspace || workspace_bytes < need)) return DT_ERR_INVALID_ARG;
            if (dt_kn7_smem_bytes(p->L, p->K, p->B, Mmax) > kSmemMax) return DT_ERR_UNSUPPORTED;
            float* table = table_on(p) ? (float*)workspace : nullptr;
            if (p->tdes) {
                const dt_tdes* q = p->tdes;
                e = dt_kn8_launch(p->batch, p->L, p->V, p->K, q->H, q->Ap, q->Ac, q->Dd, q->w, q->b0, q->s,
                                  p->root_tok, t->cand_id, table, st);
            } else if (table) {
                e = dt_kn3_table_launch(p->batch, p->L, p->V, p->K, p->R, p->U, p->Vt, p->root_tok, t->cand_id,
                                        table, st);
            }
            const float* znorm = (markov_on(p) && p->markov_norm)
                                     ? (const float*)((const unsigned char*)workspace + DT_ZNORM_OFFSET(p))
                                     : nullptr;
            if (e == cudaSuccess)
                e = dt_kn7_launch(p->batch, p->L, p->V, p->K, p->B, p->budget, Mmax, t->cand_lp, t->cand_id, table,
                                  p->root_tok,
                                  znorm, t->node_tok, t->parent, t->depth, t->rank, t->score, t->n_nodes, t->status,
                                  st);
            break;
        }
        case DT_MODE_TALON:
            if (dt_kn4_smem_bytes(kc_of(p), p->N) > kSmemMax) return DT_ERR_UNSUPPORTED;
            e = dt_kn4_launch(p->batch, p->L, kc_of(p), p->talon_k, p->log_mu, p->N, Mmax, t->cand_lp, t->cand_id,
                              t->lse, t->node_tok, t->parent, t->depth, t->rank, t->score, t->n_nodes, t->status,
                              mask, pos, pos_offset, st);
            break;
    }
    if (e == cudaSuccess && mask_out && !fuse)
        e = dt_kn5_launch(p->batch, t->L, Mmax, pos_offset, t->parent, t->depth, t->n_nodes, mask_out, pos_out,
                          t->status, st);
    return cuda_status(e);
}

dt_status dt_select(const dt_build_params* p, dt_tree* t, void* workspace, size_t workspace_bytes,
                    dt_stream_t stream) {
    return select_impl(p, t, workspace, workspace_bytes, nullptr, nullptr, 0, (cudaStream_t)stream);
}

dt_status dt_select_mask(const dt_build_params* p, dt_tree* t, void* workspace, size_t workspace_bytes,
                         int32_t pos_offset, uint32_t* mask, int32_t* pos, dt_stream_t stream) {
    if (!mask || !pos) return DT_ERR_INVALID_ARG;
    return select_impl(p, t, workspace, workspace_bytes, mask, pos, pos_offset, (cudaStream_t)stream);
}

dt_status dt_build_tree_mask(const dt_build_params* p, const void* draft_logits, dt_tree* t, void* workspace,
                             size_t workspace_bytes, int32_t pos_offset, uint32_t* mask, int32_t* pos,
                             dt_stream_t stream) {
    dt_status s = check_build(p, t);
    if (s != DT_OK) return s;
    if (!mask || !pos) return DT_ERR_INVALID_ARG;
    {
        const size_t need = dt_workspace_size(p, nullptr);
        if (need > 0 && (!workspace || workspace_bytes < need)) return DT_ERR_INVALID_ARG;
    }
    s = dt_candidates(p, draft_logits, t, stream);
    if (s != DT_OK) return s;
    if (markov_on(p) && p->markov_norm) {
        s = dt_markov_norm(p, draft_logits, t, workspace, workspace_bytes, stream);
        if (s != DT_OK) return s;
    }
    return select_impl(p, t, workspace, workspace_bytes, mask, pos, pos_offset, (cudaStream_t)stream);
}

dt_status dt_markov_norm(const dt_build_params* p, const void* draft_logits, dt_tree* t, void* workspace,
                         size_t workspace_bytes, dt_stream_t stream) {
    dt_status s = check_build(p, t);
    if (s != DT_OK) return s;
    if (!markov_on(p) || !p->markov_norm || !draft_logits) return DT_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < dt_workspace_size(p, nullptr)) return DT_ERR_INVALID_ARG;
    if ((uintptr_t)workspace & 15u) return DT_ERR_INVALID_ARG;  // the scratch tiles are bulk-copied
    unsigned char* ws = (unsigned char*)workspace;
    float* z = (float*)(ws + DT_ZNORM_OFFSET(p));
    void* scratch = ws + DT_ZNORM_OFFSET(p) + znorm_bytes(p);
    cudaError_t e = dt_kn3n_launch(draft_logits, p->dtype, p->batch, p->L, p->K, p->V, p->root_tok, t->cand_id, t->lse,
                                   p->U, p->Vt, scratch, z, (cudaStream_t)stream);
    return cuda_status(e);
}

dt_status dt_build_tree(const dt_build_params* p, const void* draft_logits, dt_tree* t, void* workspace,
                        size_t workspace_bytes, dt_stream_t stream) {
    dt_status s = check_build(p, t);
    if (s != DT_OK) return s;
    {
        const size_t need = dt_workspace_size(p, nullptr);
        if (need > 0 && (!workspace || workspace_bytes < need)) return DT_ERR_INVALID_ARG;
    }
    s = dt_candidates(p, draft_logits, t, stream);
    if (s != DT_OK) return s;
    if (markov_on(p) && p->markov_norm) {
        s = dt_markov_norm(p, draft_logits, t, workspace, workspace_bytes, stream);
        if (s != DT_OK) return s;
    }
    return dt_select(p, t, workspace, workspace_bytes, stream);
}

dt_status dt_tree_mask(const dt_tree* t, int32_t batch, int32_t pos_offset, uint32_t* mask, int32_t* pos,
                       dt_stream_t stream) {
    if (!t || !mask || !pos || batch < 1) return DT_ERR_INVALID_ARG;
    if (t->max_nodes < 1 || t->max_nodes > DT_MAX_NODES || t->L < 1 || t->L > DT_MAX_L) return DT_ERR_INVALID_ARG;
    if (!t->parent || !t->depth || !t->n_nodes || !t->status) return DT_ERR_INVALID_ARG;
    cudaError_t e = dt_kn5_launch(batch, t->L, t->max_nodes, pos_offset, t->parent, t->depth, t->n_nodes, mask, pos,
                                  t->status, (cudaStream_t)stream);
    return cuda_status(e);
}

dt_status dt_verify(const dt_tree* t, int32_t batch, int32_t V, int32_t dtype, const void* target_logits,
                    const float* target_lse, const void* draft_logits, float temperature, const float* uniforms,
                    int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok, float* visited_lse,
                    dt_stream_t stream) {
    if (temperature != 0.0f && temperature != 1.0f) return DT_ERR_UNSUPPORTED;
    return dt_verify_rule(t, batch, V, dtype, target_logits, target_lse, draft_logits,
                          temperature == 1.0f ? DT_VERIFY_RATIO : DT_VERIFY_GREEDY, uniforms, acc_nodes, acc_len,
                          next_tok, visited_lse, stream);
}

}  // extern "C"

// The walk for every rule; prop (rule DT_KN6_RATIO_MARKOV only) describes the
// normalised DARTree proposal.
static dt_status verify_impl(const dt_tree* t, int32_t batch, int32_t V, int32_t dtype, const void* target_logits,
                             const float* target_lse, const void* draft_logits, int32_t rule, const float* uniforms,
                             int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok, float* visited_lse,
                             const DtKn6Proposal* prop, cudaStream_t stream) {
    if (!t || batch < 1 || V < 1 || !target_logits || !acc_nodes || !acc_len || !next_tok) return DT_ERR_INVALID_ARG;
    if (V > DT_MAX_V) return DT_ERR_UNSUPPORTED;
    if (dtype != DT_BF16 && dtype != DT_F32) return DT_ERR_INVALID_ARG;
    if (t->max_nodes < 1 || t->max_nodes > DT_MAX_NODES || t->L < 1 || t->L > DT_MAX_L) return DT_ERR_INVALID_ARG;
    if (!t->node_tok || !t->parent || !t->depth || !t->rank || !t->n_nodes || !t->status) return DT_ERR_INVALID_ARG;
    if (rule < DT_VERIFY_GREEDY || rule > DT_KN6_RATIO_MARKOV) return DT_ERR_INVALID_ARG;
    const bool t1 = rule != DT_VERIFY_GREEDY;
    const bool uses_q = rule == DT_VERIFY_RATIO || rule == DT_VERIFY_ITER_RESIDUAL || rule == DT_KN6_RATIO_MARKOV;
    if (t1 && !uniforms) return DT_ERR_INVALID_ARG;
    if (uses_q && (!draft_logits || !t->lse)) return DT_ERR_INVALID_ARG;
    // the walk is sequential per request: spread each row over a cluster as
    // wide as the batch lets the device hold at once
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const int Mmax = t->max_nodes;
    const int s = cluster_for(
        V, batch, dtype,
        [&](int q) {
            // the residual-per-sibling rule wants clusters whose chunks leave room for its cache
            const int chunk = chunk_of(V, q, dtype);
            return chunk <= kChunkMax && dt_kn6_smem_bytes(chunk, esize, Mmax, rule) + 1024 <= kSmemMax &&
                   (rule != DT_VERIFY_ITER_RESIDUAL || dt_kn6_pq_cache(chunk, esize, Mmax, rule));
        },
        [&](int q, int chunk) { return max_clusters(6, dtype, q, chunk, Mmax * 8 + rule); },
        rule == DT_VERIFY_ITER_RESIDUAL);  // its cache leaves one CTA per SM: any cluster size that fits
    const int chunk = chunk_of(V, s, dtype);
    if (chunk > kChunkMax || dt_kn6_smem_bytes(chunk, esize, Mmax, rule) + 1024 > kSmemMax) return DT_ERR_UNSUPPORTED;
    cudaError_t e = dt_kn6_launch(batch, t->L, V, dtype, t->max_nodes, s, chunk, rule, t->node_tok, t->parent,
                                  t->depth, t->rank, t->n_nodes, t->lse, target_logits, t1 ? target_lse : nullptr,
                                  uses_q ? draft_logits : nullptr, uniforms, acc_nodes, acc_len, next_tok, visited_lse,
                                  t->status, prop, stream);
    return cuda_status(e);
}

extern "C" {

dt_status dt_verify_rule(const dt_tree* t, int32_t batch, int32_t V, int32_t dtype, const void* target_logits,
                         const float* target_lse, const void* draft_logits, int32_t rule, const float* uniforms,
                         int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok, float* visited_lse,
                         dt_stream_t stream) {
    if (rule < DT_VERIFY_GREEDY || rule > DT_VERIFY_TARGET_MATCH) return DT_ERR_INVALID_ARG;
    return verify_impl(t, batch, V, dtype, target_logits, target_lse, draft_logits, rule, uniforms, acc_nodes,
                       acc_len, next_tok, visited_lse, nullptr, (cudaStream_t)stream);
}

dt_status dt_verify_markov(const dt_build_params* p, const dt_tree* t, const void* target_logits,
                           const float* target_lse, const void* draft_logits, const float* znorm,
                           const float* uniforms, int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                           float* visited_lse, dt_stream_t stream) {
    if (!p || !t || !znorm) return DT_ERR_INVALID_ARG;
    if (p->R < 4 || p->R > 64 || (p->R & 3) || !p->U || !p->Vt) return DT_ERR_INVALID_ARG;
    if (((uintptr_t)p->Vt) & 15u) return DT_ERR_INVALID_ARG;
    if (p->batch < 1 || p->K < 1 || t->Kc != p->K || t->L != p->L) return DT_ERR_INVALID_ARG;
    const DtKn6Proposal prop{p->U, p->Vt, p->R, znorm, p->K, p->root_tok};
    return verify_impl(t, p->batch, p->V, p->dtype, target_logits, target_lse, draft_logits, DT_KN6_RATIO_MARKOV,
                       uniforms, acc_nodes, acc_len, next_tok, visited_lse, &prop, (cudaStream_t)stream);
}

dt_status dt_saba_budget(const dt_saba_params* q, const dt_tree* t, int32_t batch, const float* hidden, int32_t Hd,
                         const int32_t* prev_acc_len, int32_t* ring, int32_t* count, float* state, int32_t* budget,
                         dt_stream_t stream) {
    if (!q || !t || batch < 1 || !ring || !count || !state || !budget || !t->cand_lp) return DT_ERR_INVALID_ARG;
    if (t->L < 1 || t->L > DT_MAX_L || t->Kc < 1) return DT_ERR_INVALID_ARG;
    if (q->window < 1 || !(q->c_verify > 0.f) || !(q->c_fixed >= 0.f)) return DT_ERR_INVALID_ARG;
    if (q->B_min < 1 || q->B_max < q->B_min || q->B_max > DT_MAX_NODES - 1) return DT_ERR_INVALID_ARG;
    if (hidden && Hd < 1) return DT_ERR_INVALID_ARG;
    cudaError_t e = dt_kn9_launch(batch, t->L, t->Kc, t->cand_lp, hidden, Hd, prev_acc_len, ring, count, q->window,
                                  q->c_verify, q->c_fixed, q->B_min, q->B_max, state, budget, (cudaStream_t)stream);
    return cuda_status(e);
}

dt_status dt_test_wait_fault(int32_t kernels, int64_t budget_cycles) {
    if (kernels & ~(DT_PROBE_STAGE1 | DT_PROBE_WALK | DT_PROBE_NORMALISER)) return DT_ERR_INVALID_ARG;
    if (kernels && (budget_cycles < 1 || budget_cycles > DT_PROBE_MAX_BUDGET)) return DT_ERR_INVALID_ARG;
    const long long on = kernels ? (long long)budget_cycles : 0;
    cudaError_t e = dt_kn1_set_probe((kernels & DT_PROBE_STAGE1) ? on : 0);
    if (e == cudaSuccess) e = dt_kn6_set_probe((kernels & DT_PROBE_WALK) ? on : 0);
    if (e == cudaSuccess) e = dt_kn3n_set_probe((kernels & DT_PROBE_NORMALISER) ? on : 0);
    return cuda_status(e);
}

const char* dt_status_str(dt_status s) {
    switch (s) {
        case DT_OK: return "ok";
        case DT_ERR_INVALID_ARG: return "invalid argument";
        case DT_ERR_UNSUPPORTED: return "unsupported (outside this build's limits)";
        case DT_ERR_CUDA: return "CUDA launch or attribute call failed";
    }
    return "unknown status";
}

int32_t dt_version(void) { return 100; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free DARTree selection (dt_select_dartree_noalloc).
//
// Some callers cannot hand the library a device workspace: a serving process
// whose framework reserves the whole device memory budget up front (for
// weights and KV cache) and does not let libraries allocate more, or code on a
// latency-critical path where cudaMalloc/cudaFree are not allowed because they
// can synchronise the device.  For them the DARTree Markov table lives in a
// fixed file-scope device array instead of caller memory.  Limits: at most
// DT_NOALLOC_TABLE_BYTES of table (batch * L * K * K floats); CUDA places the
// array on a device when it loads this library's device code there (under
// lazy module loading: at the first library call on that device), and it
// stays there for the life of that device context.
// ---------------------------------------------------------------------------

namespace {

constexpr size_t kNoallocTableFloats = DT_NOALLOC_TABLE_BYTES / sizeof(float);

// Shared by every call on a device; it keeps the last call's contents.  Each
// call writes every table entry it later reads, so nothing needs clearing.
static __device__ __align__(256) float g_noalloc_table[kNoallocTableFloats];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
struct NoallocSlot {
    float* addr;               // device address of the array in that context
    unsigned long long ctx;    // the context it was looked up in (0: unknown)
};
NoallocSlot g_noalloc_slot[kNoallocMaxDevices];

// The driver's cuCtxGetId, fetched through the runtime (no link against the
// driver library); null when the driver does not offer it.
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);
CtxGetIdFn ctx_get_id_fn() {
    static CtxGetIdFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return (CtxGetIdFn)f;
    }();
    return fn;
}

// Id of the calling thread's current context; false if there is none yet.
bool current_ctx_id(unsigned long long* id) {
    CtxGetIdFn fn = ctx_get_id_fn();
    return fn && fn(nullptr, id) == 0 && *id != 0;
}

// Device address of g_noalloc_table on the current device.  Looked up with
// cudaGetSymbolAddress (which also makes the device's primary context current
// on this thread) on the first call on a device and again whenever the
// device's context has changed since (a cudaDeviceReset ends a context, and
// the address of the array in the next one may differ); otherwise cached.
dt_status noalloc_table(float** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kNoallocMaxDevices) return DT_ERR_UNSUPPORTED;
    unsigned long long ctx = 0;
    const bool have_ctx = current_ctx_id(&ctx);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot& slot = g_noalloc_slot[dev];
    if (!slot.addr || !have_ctx || slot.ctx != ctx) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_table);
        if (e != cudaSuccess || !ptr) return cuda_status(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
        slot.addr = (float*)ptr;
        slot.ctx = current_ctx_id(&ctx) ? ctx : 0;
    }
    *out = slot.addr;
    return DT_OK;
}

}  // namespace

extern "C" dt_status dt_select_dartree_noalloc(const dt_build_params* p, dt_tree* t, dt_stream_t stream) {
    dt_status s = check_build(p, t);
    if (s != DT_OK) return s;
    if (p->mode != DT_MODE_DARTREE) return DT_ERR_INVALID_ARG;
    if (p->markov_norm) return DT_ERR_UNSUPPORTED;  // the normaliser table needs caller workspace
    const bool term = p->R > 0 && p->U;
    float* table = nullptr;
    if (term) {
        const size_t need = (size_t)p->batch * p->L * p->K * p->K;
        if (need > kNoallocTableFloats) return DT_ERR_UNSUPPORTED;
        s = noalloc_table(&table);
        if (s != DT_OK) return s;
    }
    cudaError_t e = dt_kn3_launch(p->batch, p->L, p->V, p->K, dartree_w(p), p->budget_policy == DT_BUDGET_UNIFORM,
                                  p->B, p->beta, term ? p->R : 0, p->U, p->Vt,
                                  p->root_tok, t->max_nodes, t->cand_lp, t->cand_id, t->lse, table, nullptr, t->node_tok,
                                  t->parent, t->depth, t->rank, t->score, t->n_nodes, t->status, nullptr, nullptr, 0,
                                  (cudaStream_t)stream);
    return cuda_status(e);
}
