// dt_launch.h -- host-side launchers of the draft-tree kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

// Launch configuration shared by every kernel: programmatic stream
// serialisation (the kernel may start while its predecessor finishes; it
// calls griddepcontrol.wait before reading inputs) and an optional cluster.
struct DtLaunch {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    DtLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_x = 0) {
        cfg = cudaLaunchConfig_t{};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        int n = 0;
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
        if (cluster_x > 0) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = cluster_x;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = n;
    }
};

// Clusters of cluster_x CTAs of `kernel` (block threads, smem dynamic shared
// bytes; its attributes already set) that the device holds at once; 0 when the
// query fails.
template <typename K>
inline int dt_max_active_clusters(K kernel, int cluster_x, int block, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    cfg.gridDim = dim3(cluster_x, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cluster_x;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Timeout-path test hook: probe budgets (SM clock cycles, 0 = off) of the
// kernels with bounded mbarrier waits (see dt_probe_wait); synchronous.
cudaError_t dt_kn1_set_probe(long long budget);
cudaError_t dt_kn6_set_probe(long long budget);
cudaError_t dt_kn3n_set_probe(long long budget);

// Stage 1 (kn1_candidates.cu).
// grid_rows clusters share the rows round-robin.
int dt_kn1_max_clusters(int dtype, int S, int chunk, int Kc);
size_t dt_kn1_smem_bytes(int chunk, int Kc, int esize);
cudaError_t dt_kn1_launch(const void* logits, int dtype, int rows, int grid_rows, int V, int Kc, int S, int chunk,
                          float* lse, int32_t* cand_id, float* cand_lp, cudaStream_t st);

// The read floor of the cluster stage-1 launch (kn0_ceiling.cu): the same
// grid, chunks and shared memory, each CTA's chunk maximum to out[row][S].
cudaError_t dt_kn0_launch(const void* logits, int dtype, int rows, int V, int Kc, int S, int chunk, float* out,
                          int32_t* timed_out, cudaStream_t st);

// Stage 1 for many rows, one CTA per row (kn1b_rows.cu).
size_t dt_kn1b_smem_bytes();
cudaError_t dt_kn1b_launch(const void* logits, int dtype, int rows, int V, int Kc, float* lse, int32_t* cand_id,
                           float* cand_lp, cudaStream_t st);

// DDTree selection (kn2_ddtree.cu).
size_t dt_kn2_smem_bytes(int L, int K, int B);
// budget: NULL, or [batch] per-request budgets clamped to [1, B] (B sizes the buffers).
cudaError_t dt_kn2_launch(int batch, int L, int K, int B, const int32_t* budget, int Mmax, const float* cand_lp,
                          const int32_t* cand_id,
                          const float* lse, int32_t* tok, int32_t* parent, int32_t* depth, int32_t* rank,
                          float* score, int32_t* n_nodes, int32_t* status, uint32_t* mask, int32_t* pos,
                          int pos_offset, cudaStream_t st);

// DARTree Markov table + selection (kn3_dartree.cu).
size_t dt_kn3_table_smem_bytes(int K, int R);
size_t dt_kn3_select_smem_bytes(int L, int K, int W, int use_table);
// wfix = 1: per-depth widths B/L (+1 for the first B%L depths), W their maximum.
cudaError_t dt_kn3_launch(int batch, int L, int V, int K, int W, int wfix, int B, float beta, int R, const float* U,
                          const float* Vt, const int32_t* root_tok, int Mmax, const float* cand_lp,
                          const int32_t* cand_id, const float* lse, float* table, const float* znorm, int32_t* tok,
                          int32_t* parent, int32_t* depth, int32_t* rank, float* score, int32_t* n_nodes,
                          int32_t* status, uint32_t* mask, int32_t* pos, int pos_offset, cudaStream_t st);

// The Markov edge table alone, [batch][L][K][K] (row 0 of position 0: the
// root token, left unwritten without one).
cudaError_t dt_kn3_table_launch(int batch, int L, int V, int K, int R, const float* U, const float* Vt,
                                const int32_t* root_tok, const int32_t* cand_id, float* table, cudaStream_t st);

// Best-first heap with parent-conditioned edge scores (kn7_heap.cu): edge
// terms from `table` ([batch][L][K][K], or NULL: none), minus znorm when given;
// the depth-1 term only when root_tok names a token.  Returns
// cudaErrorInvalidValue when the shapes do not fit shared memory.
size_t dt_kn7_smem_bytes(int L, int K, int B, int Mmax);
cudaError_t dt_kn7_launch(int batch, int L, int V, int K, int B, const int32_t* budget, int Mmax, const float* cand_lp,
                          const int32_t* cand_id, const float* table, const int32_t* root_tok, const float* znorm,
                          int32_t* tok, int32_t* parent, int32_t* depth, int32_t* rank, float* score,
                          int32_t* n_nodes, int32_t* status, cudaStream_t st);

// TDES edge table (kn7_heap.cu): [batch][L][K][K] = s * f(parent, child, depth).
size_t dt_kn8_smem_bytes(int K, int H);
cudaError_t dt_kn8_launch(int batch, int L, int V, int K, int H, const float* Ap, const float* Ac, const float* Dd,
                          const float* w, float b0, float s, const int32_t* root_tok, const int32_t* cand_id,
                          float* table, cudaStream_t st);

// SABA state and per-request budgets (kn9_saba.cu).
cudaError_t dt_kn9_launch(int batch, int L, int Kc, const float* cand_lp, const float* hidden, int Hd,
                          const int32_t* prev_len, int32_t* ring, int32_t* count, int w, float c_verify,
                          float c_fixed, int B_min, int B_max, float* state, int32_t* budget, cudaStream_t st);

// TALON selection (kn4_talon.cu).
size_t dt_kn4_smem_bytes(int Kc, int N);
cudaError_t dt_kn4_launch(int batch, int L, int Kc, int talon_k, float log_mu, int N, int Mmax,
                          const float* cand_lp, const int32_t* cand_id, const float* lse, int32_t* tok,
                          int32_t* parent, int32_t* depth, int32_t* rank, float* score, int32_t* n_nodes,
                          int32_t* status, uint32_t* mask, int32_t* pos, int pos_offset, cudaStream_t st);

// Full-vocabulary DARTree log-normalisers on the tensor cores (kn3n_norm.cu):
// z [batch][L][K]; scratch: 256-byte aligned, dt_kn3n_scratch_bytes(batch * L * K, V)
// bytes (per-slice partial sums, then the child-token table in bf16).
#define DT_KN3N_MAX_SPLIT 256
size_t dt_kn3n_scratch_bytes(int rows, int V);
cudaError_t dt_kn3n_launch(const void* x, int dtype, int batch, int L, int K, int V, const int32_t* root_tok,
                           const int32_t* cand_id, const float* lse, const float* U, const float* Vt, void* scratch,
                           float* z, cudaStream_t st);

// Tree mask (kn5_mask.cu).
size_t dt_kn5_smem_bytes(int Mmax);
cudaError_t dt_kn5_launch(int batch, int L, int Mmax, int pos_offset, const int32_t* parent, const int32_t* depth,
                          const int32_t* n_nodes, uint32_t* mask, int32_t* pos, int32_t* status, cudaStream_t st);

// Verification walk (kn6_verify.cu); rule: DT_VERIFY_*, or DT_KN6_RATIO_MARKOV:
// the ratio rule against the normalised DARTree proposal described by `prop`.
#define DT_KN6_RATIO_MARKOV 4
struct DtKn6Proposal {
    const float* U;           // [V][R] fp32
    const float* Vt;          // [V][R] fp32, 16-byte aligned
    int R;                    // 4..64, a multiple of 4
    const float* z;           // [batch][L][K] log-normalisers
    int K;
    const int32_t* root_tok;  // [batch] or NULL
};
int dt_kn6_max_clusters(int dtype, int S, int chunk, int Mmax, int rule);
size_t dt_kn6_smem_bytes(int chunk, int esize, int Mmax, int rule);
int dt_kn6_pq_cache(int chunk, int esize, int Mmax, int rule);  // 1: the residual passes cache (P, Q)
cudaError_t dt_kn6_launch(int batch, int L, int V, int dtype, int Mmax, int S, int chunk, int rule,
                          const int32_t* tok, const int32_t* parent, const int32_t* depth, const int32_t* rank,
                          const int32_t* n_nodes, const float* draft_lse, const void* target,
                          const float* target_lse, const void* draft,
                          const float* uniforms, int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                          float* visited_lse, int32_t* status, const DtKn6Proposal* prop, cudaStream_t st);
