// kn3_dartree.cu -- DARTree depth-wise supertree and deferred Top-B pruning.
//
// [DARTree] Algorithm 1: per depth d, score every child (one of the
// position's Top-K tokens) of every kept parent with the causal correction,
// s(child) = (s(parent) + log q~_d) + beta, keep the W best children of all
// parents, accumulate them into the supertree S; finally T = TopB(S).
// "Deferred best-first pruning":
// s_beta = sum log q~ + beta*d; Lemma 1: with beta <= 0 and every log q~ <= 0,
// TopB(S) equals the best-first heap over S.
//
// The correction head is a parent-conditioned Markov term on the candidates,
// log q~_d(c | u) = lp_d(c) + <U[tok(u)], Vt[c]>, the dot product a serial fp32
// fma chain over R (bit-reproducible).  Kernel A computes, per request and
// position, the K x K table of these terms for every (parent rank, child
// rank) pair of consecutive positions (the parents of depth-d nodes are always
// among position d-1's candidates) into the caller's workspace.  Kernel B, one
// CTA per request, builds S in shared memory depth by depth (W*K candidates,
// bitonic sort on (score, lexicographic position) keys), ranks all of S in the
// shared node order by merging the per-depth sorted layers, and emits TopB(S)
// when it is topologically ordered; otherwise (some edge raised the score) it
// runs the best-first heap over S and sets DT_DEV_BESTFIRST.
// DARTree (fixed) (wfix): depth d keeps B / L children, one more for each of the
// first B mod L depths (the shallowest), instead of W; the widths sum to B, so
// the final pruning keeps all of S.
#include "dt_device.cuh"
#include "dt_mask.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT_TAB = 256;
constexpr int NT = 512;

// ---- kernel A: Markov table ------------------------------------------------
__global__ void __launch_bounds__(NT_TAB) kn3_table_kernel(int L, int K, int R, int V, const float* __restrict__ U,
                                                           const float* __restrict__ Vt,
                                                           const int32_t* __restrict__ root_tok,
                                                           const int32_t* __restrict__ cand_id,
                                                           float* __restrict__ table) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int d = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int Rp = R | 1;  // odd row stride: conflict-free column reads
    dt_pdl_trigger();
    dt_pdl_wait();
    float* Us = (float*)smem;
    float* Vs = Us + (size_t)K * Rp;
    int np;
    if (d == 0) {
        const int rt = root_tok ? root_tok[b] : -1;
        if (rt < 0 || rt >= V) return;  // no term at depth 1
        np = 1;
        for (int k = tid; k < R; k += NT_TAB) Us[k] = U[(size_t)rt * R + k];
    } else {
        np = K;
        for (int t = tid; t < K * R; t += NT_TAB) {
            const int i = t / R, k = t % R;
            const int tok = cand_id[((size_t)b * L + d - 1) * K + i];
            Us[i * Rp + k] = U[(size_t)tok * R + k];
        }
    }
    for (int t = tid; t < K * R; t += NT_TAB) {
        const int j = t / R, k = t % R;
        const int tok = cand_id[((size_t)b * L + d) * K + j];
        Vs[j * Rp + k] = Vt[(size_t)tok * R + k];
    }
    __syncthreads();
    float* out = table + ((size_t)b * L + d) * K * K;
    for (int t = tid; t < np * K; t += NT_TAB) {
        const int i = t / K, j = t % K;
        const float* u = Us + (size_t)i * Rp;
        const float* v = Vs + (size_t)j * Rp;
        float acc = 0.f;
        for (int k = 0; k < R; ++k) acc = __fmaf_rn(u[k], v[k], acc);
        out[i * K + j] = acc;
    }
}

// ---- kernel B: supertree + deferred Top-B -----------------------------------
struct Kn3Smem {
    unsigned long long* cand;  // [pow2(W*K)] candidate keys; reused for lexicographic sorts
    float* lp;                 // [K]
    float* s;                  // [W*L] supertree nodes
    int* dep;
    int* par;
    int* rank;
    uint32_t* lex;
    int* grank;   // [W*L] position in the node order
    int* lexl;    // [W] previous layer in lexicographic order
    int* order;   // [W*L] output order / heap
    int* cstart;  // [W*L + 1] children CSR (fallback)
    int* clist;   // [W*L]
    unsigned long long* scratch;  // [NT] warp-list merges (W <= 32)
    float* lps;   // [L*K] the request's candidate log-probs
    float* tabs;  // [L*K*K] the request's Markov table, when it fits (else nullptr)
    float* zs;    // [L*K] the request's log-normalisers (normalised correction)
};

// Markov table entries staged in shared memory per request, at most.
constexpr int kTabStage = 16384;

DT_DI size_t kn3_cap(int W, int K) { return (size_t)dt_pow2_ceil(W * K > W ? W * K : W); }

DT_DI Kn3Smem kn3_carve(unsigned char* p, int L, int K, int W, bool stage_tab) {
    Kn3Smem m;
    const int NS = W * L;
    m.scratch = (unsigned long long*)p;
    p += (size_t)NT * 8;
    m.lps = (float*)p;
    p += (size_t)((L * K + 3) & ~3) * 4;
    m.zs = (float*)p;
    p += (size_t)((L * K + 3) & ~3) * 4;
    m.tabs = nullptr;
    if (stage_tab) {
        m.tabs = (float*)p;
        p += (size_t)L * K * K * 4;
    }
    m.cand = (unsigned long long*)p;
    p += kn3_cap(W, K) * 8;
    m.lp = (float*)p; p += (size_t)((K + 3) & ~3) * 4;
    m.s = (float*)p; p += (size_t)NS * 4;
    m.dep = (int*)p; p += (size_t)NS * 4;
    m.par = (int*)p; p += (size_t)NS * 4;
    m.rank = (int*)p; p += (size_t)NS * 4;
    m.lex = (uint32_t*)p; p += (size_t)NS * 4;
    m.grank = (int*)p; p += (size_t)NS * 4;
    m.order = (int*)p; p += (size_t)NS * 4;
    m.clist = (int*)p; p += (size_t)NS * 4;
    m.cstart = (int*)p; p += (size_t)(NS + 1) * 4;
    m.lexl = (int*)p;
    return m;
}

// The node order made total for any scores: scores compare by their order
// keys (so a NaN has a place), equal keys by dt_node_before, and a pair that
// neither precedes (only NaN scores do that) by node index.  For finite
// scores it is dt_node_before.
DT_DI bool node_before_total(int y, int x, const float* s, const int* dep, const int* par, const uint32_t* lex) {
    const uint32_t ky = dt_fkey(s[y]), kx = dt_fkey(s[x]);
    if (ky != kx) return ky > kx;
    if (dt_node_before(y, x, s, dep, par, lex)) return true;
    if (dt_node_before(x, y, s, dep, par, lex)) return false;
    return y < x;
}

__global__ void __launch_bounds__(NT, 1) kn3_select_kernel(int L, int K, int W, int wfix, int B, float beta, int use_table,
                                                        const int32_t* __restrict__ root_tok, int V,
                                                        int Mmax, const float* __restrict__ cand_lp,
                                                        const int32_t* __restrict__ cand_id,
                                                        const float* __restrict__ lse,
                                                        const float* __restrict__ table,
                                                        const float* __restrict__ znorm,
                                                        int32_t* __restrict__ o_tok, int32_t* __restrict__ o_par,
                                                        int32_t* __restrict__ o_dep, int32_t* __restrict__ o_rank,
                                                        float* __restrict__ o_score, int32_t* __restrict__ o_n,
                                                        int32_t* __restrict__ status, uint32_t* __restrict__ o_mask,
                                                        int32_t* __restrict__ o_pos, int pos_offset) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int lay_start[DT_MAX_L + 2];
    __shared__ int sh_bad, sh_viol;
    const int b = blockIdx.x, tid = threadIdx.x;
    const bool stage_tab = use_table && L * K * K <= kTabStage;
    Kn3Smem S = kn3_carve(smem, L, K, W, stage_tab);
    dt_pdl_trigger();
    dt_pdl_wait();
    const int rt = root_tok ? root_tok[b] : -1;
    const bool term1 = use_table && rt >= 0 && rt < V;
    // the request's log-probs (and Markov table, when small) into shared memory
    for (int i = tid; i < L * K; i += NT) {
        S.lps[i] = cand_lp[(size_t)b * L * K + i];
        S.zs[i] = znorm ? znorm[(size_t)b * L * K + i] : 0.f;
    }
    if (stage_tab) {
        const float* tb = table + (size_t)b * L * K * K;
        const int n = L * K * K;
        const int n4 = (((uintptr_t)tb & 15u) == 0) ? n / 4 : 0;  // 16-byte loads where aligned
        for (int i = tid; i < n4; i += NT) ((float4*)S.tabs)[i] = ((const float4*)tb)[i];
        for (int i = n4 * 4 + tid; i < n; i += NT) S.tabs[i] = tb[i];
    }
    __syncthreads();

    int nS = 0;      // supertree nodes so far
    int nprev = 1;   // size of the previous layer (the root)
    if (tid == 0) { lay_start[0] = 0; sh_bad = 0; sh_viol = 0; }
    for (int d = 1; d <= L; ++d) {
        const float* lpd = S.lps + (size_t)(d - 1) * K;
        const bool term = use_table && (d > 1 || term1);
        const float* tab = !term ? nullptr
                                 : (stage_tab ? S.tabs + (size_t)(d - 1) * K * K
                                              : table + ((size_t)b * L + d - 1) * K * K);
        const int m = nprev * K;
        // key of candidate idx = (parent j in lexicographic order, child rank r)
        auto key_of = [&](int idx) {
            const int j = idx / K, r = idx % K;
            const int p = (d == 1) ? -1 : S.lexl[j];
            const float sp = (d == 1) ? 0.f : S.s[p];
            float t = lpd[r];
            if (term) {
                const int pr = (d == 1) ? 0 : S.rank[p];  // parent's candidate index (root: row 0)
                t = __fadd_rn(t, tab[(size_t)pr * K + r]);
                if (znorm) t = __fsub_rn(t, S.zs[(size_t)(d - 1) * K + pr]);  // normalised: minus log Z
            }
            const float sc = __fadd_rn(__fadd_rn(sp, t), beta);
            const uint32_t lx = ((uint32_t)j << 16) | (uint32_t)r;
            return ((unsigned long long)dt_fkey(sc) << 32) | (unsigned long long)(0xFFFFFFFFu - lx);
        };
        // layer width: W, or (DARTree fixed) B spread over the depths, the
        // remainder to the shallowest ones (W is then the largest of them)
        const int keep = min(wfix ? B / L + (d - 1 < B % L ? 1 : 0) : W, m);
        if (W <= 32) {
            // top-W: warp sorts merged in a tree; the layer's lexicographic
            // order by warp 0 alone
            const unsigned long long y = dt_block_top32<NT>(m, key_of, S.scratch);
            if (tid < 32) {
                uint32_t lx = 0;
                int par = -1;
                if (tid < keep) {
                    lx = 0xFFFFFFFFu - (uint32_t)y;
                    const int j = (int)(lx >> 16), r = (int)(lx & 0xFFFFu);
                    const int x = nS + tid;
                    par = (d == 1) ? -1 : S.lexl[j];
                    S.s[x] = dt_fkey_val((uint32_t)(y >> 32));
                    S.dep[x] = d;
                    S.par[x] = par;
                    S.rank[x] = r;
                    S.lex[x] = lx;
                }
                __syncwarp();  // every lane has read lexl before it is rewritten
                const unsigned long long k2 =
                    dt_warp_sort_reg(tid < keep ? (((unsigned long long)lx << 32) | (unsigned)(nS + tid)) : ~0ull, false);
                if (tid < keep) S.lexl[tid] = (int)(k2 & 0xFFFFFFFFull);
            }
        } else {
            const int P2 = dt_pow2_ceil(m);
            for (int idx = tid; idx < P2; idx += NT) S.cand[idx] = idx < m ? key_of(idx) : 0ull;
            __syncthreads();
            dt_bitonic_u64<NT>(S.cand, P2, true);
            for (int q = tid; q < keep; q += NT) {
                const unsigned long long y = S.cand[q];
                const uint32_t lx = 0xFFFFFFFFu - (uint32_t)y;
                const int j = (int)(lx >> 16), r = (int)(lx & 0xFFFFu);
                const int x = nS + q;
                S.s[x] = dt_fkey_val((uint32_t)(y >> 32));
                S.dep[x] = d;
                S.par[x] = (d == 1) ? -1 : S.lexl[j];
                S.rank[x] = r;
                S.lex[x] = lx;
            }
            __syncthreads();
            // previous-layer order for the next depth: this layer by lexicographic key
            const int Q2 = dt_pow2_ceil(keep);
            for (int q = tid; q < Q2; q += NT)
                S.cand[q] = (q < keep) ? (((unsigned long long)S.lex[nS + q] << 32) | (unsigned)(nS + q)) : ~0ull;
            __syncthreads();
            dt_bitonic_u64<NT>(S.cand, Q2, false);
            for (int q = tid; q < keep; q += NT) S.lexl[q] = (int)(S.cand[q] & 0xFFFFFFFFull);
        }
        __syncthreads();
        nS += keep;
        nprev = keep;
        if (tid == 0) lay_start[d] = nS;
    }
    __syncthreads();

    // edges whose child outscores its parent (Lemma 1 needs none); counted
    // per warp first -- hundreds of atomics on one word would serialise
    {
        int nv = 0;
        for (int x = tid; x < nS; x += NT) {
            const int p = S.par[x];
            const float sp = p < 0 ? 0.f : S.s[p];
            nv += S.s[x] > sp;
        }
        nv = dt_warp_sum_i(nv);
        if ((tid & 31) == 0 && nv) atomicAdd(&sh_viol, nv);
    }
    // rank of every node in the shared order: a merge tree over the per-depth
    // layers, each sorted in that order and stored contiguously.  At level l
    // lists of 2^l layers merge pairwise: an element's place in the merged
    // list is its place in its own list plus the partner list's elements
    // before it (one binary search; score keys decide unless equal, then the
    // full node order).  cur[p] is the node at position p; the merged lists
    // keep the layers' position ranges.
    {
        int* cur = S.order;
        int* nxt = S.clist;
        for (int x = tid; x < nS; x += NT) cur[x] = x;
        __syncthreads();
        // a strict total order whatever the scores (NaN included): positions
        // of the merged lists are then a permutation
        auto before = [&](int y, int x, uint32_t kx) {
            const uint32_t ky = dt_fkey(S.s[y]);
            if (ky != kx) return ky > kx;
            return node_before_total(y, x, S.s, S.dep, S.par, S.lex);
        };
        // (an entry is read clamped into [0, nS): a defence that keeps every
        // index inside the tree should the order ever not be total)
        auto node_at = [&](int q) { const int v = cur[q]; return (unsigned)v < (unsigned)nS ? v : 0; };
        for (int w = 1; w < L; w <<= 1) {  // list width in layers
            for (int p = tid; p < nS; p += NT) {
                const int x = node_at(p);
                const uint32_t kx = dt_fkey(S.s[x]);
                const int li = (S.dep[x] - 1) / w;  // list index
                const int A = li & ~1;              // the pair's first list
                const int a0 = lay_start[min(A * w, L)], b0 = lay_start[min((A + 1) * w, L)];
                const int b1 = lay_start[min((A + 2) * w, L)];
                int lo, hi;
                if (li == A) {
                    lo = b0;
                    hi = b1;
                } else {
                    lo = a0;
                    hi = b0;
                }
                const int base = lo;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (before(node_at(mid), x, kx)) lo = mid + 1;
                    else hi = mid;
                }
                const int j = lo - base;
                const int np = li == A ? p + j : p - (b0 - a0) + j;
                if ((unsigned)np < (unsigned)nS) nxt[np] = x;
            }
            __syncthreads();
            int* t = cur;
            cur = nxt;
            nxt = t;
        }
        for (int p = tid; p < nS; p += NT) S.grank[node_at(p)] = p;
        __syncthreads();
    }
    const int nT = min(B, nS);
    for (int x = tid; x < nS; x += NT) {
        const int g = S.grank[x];
        if (g < nT) {
            S.order[g] = x;
            const int p = S.par[x];
            if (p >= 0 && S.grank[p] >= g) sh_bad = 1;  // TopB(S) is not a tree in topological order
        }
    }
    __syncthreads();

    const size_t ob = (size_t)b * Mmax;
    if (sh_bad) {
        // best-first heap over S from the root's children (single thread; only
        // reachable when some edge raises the score)
        for (int x = tid; x <= nS; x += NT) S.cstart[x] = 0;
        __syncthreads();
        for (int x = tid; x < nS; x += NT)
            if (S.par[x] >= 0) atomicAdd(&S.cstart[S.par[x] + 1], 1);
        __syncthreads();
        if (tid == 0) {
            for (int x = 0; x < nS; ++x) S.cstart[x + 1] += S.cstart[x];
            for (int x = 0; x < nS; ++x) S.grank[x] = S.cstart[x];  // fill cursors
            for (int x = 0; x < nS; ++x)
                if (S.par[x] >= 0) S.clist[S.grank[S.par[x]]++] = x;
            // heap in S.grank[] (cursors no longer needed), output order in S.order[]
            int* heap = S.grank;
            int hn = 0;
            auto push = [&](int v) {
                int i = hn++;
                heap[i] = v;
                while (i > 0) {
                    const int pi = (i - 1) >> 1;
                    if (!dt_node_before(heap[i], heap[pi], S.s, S.dep, S.par, S.lex)) break;
                    const int t = heap[i]; heap[i] = heap[pi]; heap[pi] = t;
                    i = pi;
                }
            };
            auto pop = [&]() {
                const int top = heap[0];
                heap[0] = heap[--hn];
                int i = 0;
                for (;;) {
                    const int l = 2 * i + 1, r = l + 1;
                    int bi = i;
                    if (l < hn && dt_node_before(heap[l], heap[bi], S.s, S.dep, S.par, S.lex)) bi = l;
                    if (r < hn && dt_node_before(heap[r], heap[bi], S.s, S.dep, S.par, S.lex)) bi = r;
                    if (bi == i) break;
                    const int t = heap[i]; heap[i] = heap[bi]; heap[bi] = t;
                    i = bi;
                }
                return top;
            };
            for (int x = 0; x < lay_start[1]; ++x) push(x);
            int n = 0;
            while (n < B && hn > 0) {
                const int x = pop();
                S.order[n++] = x;
                for (int c = S.cstart[x]; c < S.cstart[x + 1]; ++c) push(S.clist[c]);
            }
            sh_bad = n;  // nodes emitted
        }
        __syncthreads();
    }
    const int nOut = sh_bad ? sh_bad : nT;
    // output index of every supertree node (reuse cstart as a map)
    for (int x = tid; x < nS; x += NT) S.cstart[x] = -1;
    __syncthreads();
    for (int q = tid; q < nOut; q += NT) S.cstart[S.order[q]] = q + 1;
    __syncthreads();
    for (int q = tid; q < nOut; q += NT) {
        const int x = S.order[q];
        const int dd = S.dep[x], rr = S.rank[x], p = S.par[x];
        o_tok[ob + q + 1] = cand_id[((size_t)b * L + dd - 1) * K + rr];
        o_par[ob + q + 1] = p < 0 ? 0 : S.cstart[p];
        o_dep[ob + q + 1] = dd;
        o_rank[ob + q + 1] = rr;
        o_score[ob + q + 1] = S.s[x];
        if (o_mask) o_pos[ob + q + 1] = dd + pos_offset;
    }
    if (tid == 0) {
        if (o_mask) o_pos[ob] = pos_offset;
        o_tok[ob] = -1;
        o_par[ob] = -1;
        o_dep[ob] = 0;
        o_rank[ob] = -1;
        o_score[ob] = 0.f;
        o_n[b] = nOut + 1;
        int bits = sh_bad ? DT_DEV_BESTFIRST : 0;
        const int v = sh_viol < (1 << 23) - 1 ? sh_viol : (1 << 23) - 1;
        bits |= v << DT_DEV_VIOLATION_SHIFT;
        for (int l = 0; l < L; ++l) {
            const float x = lse[(size_t)b * L + l];
            if (x != x) bits |= DT_DEV_TIMEOUT;  // stage 1 flagged this row
        }
        if (znorm)
            for (int i = 0; i < L * K; ++i)
                if (S.zs[i] != S.zs[i]) bits |= DT_DEV_TIMEOUT;  // the normaliser kernel flagged this row
        status[b] = bits;
    }
    if (o_mask) {  // fused tree mask (positions above): parents through the output map in shared memory
        dt_write_mask_rows<NT>(nOut + 1, Mmax,
                               [&](int a) {
                                   if (a == 0) return -1;
                                   const int p = S.par[S.order[a - 1]];
                                   return p < 0 ? 0 : S.cstart[p];
                               },
                               o_mask + (size_t)b * Mmax * ((Mmax + 31) >> 5));
    }
}

}  // namespace

size_t dt_kn3_table_smem_bytes(int K, int R) { return (size_t)2 * K * (R | 1) * 4 + 16; }

size_t dt_kn3_select_smem_bytes(int L, int K, int W, int use_table) {
    int cap = 1;
    while (cap < W * K || cap < W) cap <<= 1;
    const size_t NS = (size_t)W * L;
    const bool stage_tab = use_table && L * K * K <= kTabStage;
    return (size_t)NT * 8 + (size_t)((L * K + 3) & ~3) * 8 + (stage_tab ? (size_t)L * K * K * 4 : 0) +
           (size_t)cap * 8 + (size_t)((K + 3) & ~3) * 4 + NS * 4 * 8 + (NS + 1) * 4 + (size_t)W * 4 + 16;
}

cudaError_t dt_kn3_table_launch(int batch, int L, int V, int K, int R, const float* U, const float* Vt,
                                const int32_t* root_tok, const int32_t* cand_id, float* table, cudaStream_t st) {
    const size_t sm = dt_kn3_table_smem_bytes(K, R);
    cudaError_t e = cudaFuncSetAttribute(kn3_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    DtLaunch lt(dim3(L, batch), dim3(NT_TAB), sm, st);
    return cudaLaunchKernelEx(&lt.cfg, kn3_table_kernel, L, K, R, V, U, Vt, root_tok, cand_id, table);
}

cudaError_t dt_kn3_launch(int batch, int L, int V, int K, int W, int wfix, int B, float beta, int R, const float* U,
                          const float* Vt, const int32_t* root_tok, int Mmax, const float* cand_lp,
                          const int32_t* cand_id, const float* lse, float* table, const float* znorm, int32_t* tok,
                          int32_t* parent, int32_t* depth, int32_t* rank, float* score, int32_t* n_nodes,
                          int32_t* status, uint32_t* mask, int32_t* pos, int pos_offset, cudaStream_t st) {
    cudaError_t e;
    const int use_table = (R > 0 && table != nullptr) ? 1 : 0;
    if (use_table) {
        const size_t sm = dt_kn3_table_smem_bytes(K, R);
        if ((e = cudaFuncSetAttribute(kn3_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) !=
            cudaSuccess)
            return e;
        DtLaunch lt(dim3(L, batch), dim3(NT_TAB), sm, st);
        if ((e = cudaLaunchKernelEx(&lt.cfg, kn3_table_kernel, L, K, R, V, U, Vt, root_tok, cand_id, table)) !=
            cudaSuccess)
            return e;
    }
    const size_t sm = dt_kn3_select_smem_bytes(L, K, W, use_table);
    if ((e = cudaFuncSetAttribute(kn3_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) !=
        cudaSuccess)
        return e;
    DtLaunch ls(dim3(batch), dim3(NT), sm, st);
    return cudaLaunchKernelEx(&ls.cfg, kn3_select_kernel, L, K, W, wfix, B, beta, use_table, root_tok, V, Mmax, cand_lp,
                              cand_id, lse, (const float*)table, znorm, tok, parent, depth, rank, score, n_nodes,
                              status, mask, pos, pos_offset);
}
