// kn6_verify.cu -- acceptance walk over the draft tree.
//
// [DARTree] "Speculative sampling": at T=0 accept draft tokens while they
// match the target's greedy choice and emit the target's choice at the first
// mismatch; at T=1 accept y ~ q with min(1, p/q) and on rejection draw one
// replacement from the normalised residual [p - q]_+.  [Unit11] worked
// three-token example (R = 0 skips the residual; p(x) = 0 < q(x) always
// rejects), bonus-token section (a node with nothing left to verify samples
// one more token from its target row), greedy ties (smallest id).
//
// On a tree (the pages give the single-chain rule): at node n the children of
// n are tested in rank order and the walk descends into the first accepted
// one; if all are rejected the replacement comes from max(0, P - Q) with P, Q
// the 2^32 fixed-point masses of the target row of n and the drafter row of
// n's children's position (P when the residual is empty); a node without
// children draws its bonus token from P.  Ratios and masses use dt_exp_canon,
// and the draw is an exact integer inverse CDF, so results are reproducible.
//
// One thread-block cluster of S CTAs per request; CTA c owns a vocabulary
// chunk.  Per visited node each CTA bulk-copies its chunk of the target row
// into shared memory (the only HBM traffic: visited rows, plus one drafter
// row on a T=1 rejection); partial argmax / (max, sum exp) / residual sums are
// combined across the cluster through distributed shared memory.
#include "dt_device.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int SMAX = 16;

struct Pub {
    float m, s;
    unsigned long long u;
};

struct Kn6Misc {
    uint64_t bar;
    int timeout;
    int bad;
    Pub pub[2];
    unsigned long long red_u[NW];
    float red_f[NW];
    int red_i[NW];
    unsigned long long scan_u[NW];
    int child;
    int nkids;
    int found_v;
};

DT_DI unsigned long long warp_max_u64(unsigned long long v) {
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long t = __shfl_xor_sync(0xffffffffu, v, o);
        v = t > v ? t : v;
    }
    return v;
}

template <typename T>
__global__ void __launch_bounds__(NT) kn6_kernel(int L, int V, int Mmax, int chunk, int t1,
                                                 const int32_t* __restrict__ g_tok,
                                                 const int32_t* __restrict__ g_par,
                                                 const int32_t* __restrict__ g_dep,
                                                 const int32_t* __restrict__ g_rank,
                                                 const int32_t* __restrict__ g_n,
                                                 const float* __restrict__ draft_lse, const T* __restrict__ target,
                                                 const float* __restrict__ target_lse,
                                                 const T* __restrict__ draft, const float* __restrict__ uniforms,
                                                 int32_t* __restrict__ acc_nodes, int32_t* __restrict__ acc_len,
                                                 int32_t* __restrict__ next_tok, float* __restrict__ visited_lse,
                                                 int32_t* __restrict__ status) {
    using E = DtElem<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int c = (int)cluster.block_rank();
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int lo = min(V, c * chunk), hi = min(V, lo + chunk);
    const int nch = hi - lo;

    Kn6Misc* misc = (Kn6Misc*)smem;
    int* s_tok = (int*)(smem + 1024);
    int* s_par = s_tok + Mmax;
    int* s_dep = s_par + Mmax;
    int* s_rank = s_dep + Mmax;
    unsigned char* dbuf = smem + 1024 + (size_t)(((Mmax * 16) + 127) & ~127);

    if (tid == 0) {
        dt_mbar_init(&misc->bar, 1);
        dt_fence_mbar_init();
        misc->timeout = 0;
    }
    dt_pdl_trigger();
    dt_pdl_wait();  // the tree and the target rows come from earlier kernels
    const int M = g_n[b];
    if (tid == 0) misc->bad = (M < 1 || M > Mmax) ? 1 : 0;
    __syncthreads();
    const size_t tb = (size_t)b * Mmax;
    if (!misc->bad) {
        for (int i = tid; i < M; i += NT) {
            s_tok[i] = g_tok[tb + i];
            s_par[i] = g_par[tb + i];
            s_dep[i] = g_dep[tb + i];
            s_rank[i] = g_rank[tb + i];
        }
        __syncthreads();
        for (int i = tid; i < M; i += NT) {
            const int p = s_par[i], d = s_dep[i];
            bool ok;
            if (i == 0) ok = (p == -1 && d == 0);
            else ok = (p >= 0 && p < M && p != i && d >= 1 && d <= L && d == s_dep[p] + 1 && s_tok[i] >= 0 &&
                       s_tok[i] < V);
            if (!ok) misc->bad = 1;
        }
    }
    __syncthreads();
    if (misc->bad) {  // identical decision in every CTA of the cluster: nobody syncs below
        if (c == 0 && tid == 0) {
            atomicOr(&status[b], DT_DEV_BAD_TREE);
            acc_len[b] = 0;
            next_tok[b] = -1;
        }
        if (c == 0)
            for (int i = tid; i <= L; i += NT) acc_nodes[(size_t)b * (L + 1) + i] = -1;
        return;
    }

    int n = 0, len = 0;
    uint32_t phase = 0;
    int k = 0;  // cluster exchanges so far (selects the Pub slot)
    int out_tok = -1;
    const float* u0 = uniforms ? uniforms + (size_t)b * 2 * Mmax : nullptr;
    const float* u1 = u0 ? u0 + Mmax : nullptr;

    for (;;) {
        // ---- stage this CTA's chunk of target row n -----------------------
        const T* trow = target + (tb + n) * (size_t)V;
        uint32_t bytes = 0;
        __syncthreads();
        dt_fence_proxy_async();
        const T* x = dt_stage_row<T>(trow, lo, hi, dbuf, &misc->bar, &bytes);
        if (bytes) {
            // one thread waits on the copy; the others block in the barrier
            if (tid == 0 && !dt_mbar_wait(&misc->bar, phase)) {
                misc->timeout = 1;
                dt_mbar_wait(&misc->bar, phase);
            }
            phase ^= 1;
        }
        __syncthreads();

        int child = -1;
        float lse_t = 0.f;
        if (!t1) {
            // argmax, smallest id on ties: max of (key << 32 | ~id)
            unsigned long long best = 0;
            for (int e = tid; e < nch; e += NT) {
                unsigned long long key = ((unsigned long long)E::key(x[e]) << 32) |
                                         (unsigned long long)(0xFFFFFFFFu - (uint32_t)(lo + e));
                best = key > best ? key : best;
            }
            best = warp_max_u64(best);
            if (lane == 0) misc->red_u[wid] = best;
            __syncthreads();
            if (tid == 0) {
                unsigned long long a = 0;
                for (int w = 0; w < NW; ++w) a = misc->red_u[w] > a ? misc->red_u[w] : a;
                misc->pub[k & 1].u = a;
            }
            __syncthreads();
            cluster.sync();
            unsigned long long part[SMAX];
#pragma unroll
            for (int j = 0; j < SMAX; ++j) part[j] = (j < S) ? cluster.map_shared_rank(misc, j)->pub[k & 1].u : 0ull;
            unsigned long long g = 0;
#pragma unroll
            for (int j = 0; j < SMAX; ++j) g = part[j] > g ? part[j] : g;
            ++k;
            const int a = (int)(0xFFFFFFFFu - (uint32_t)(g & 0xFFFFFFFFull));
            out_tok = a;
            if (tid == 0) misc->child = 0x7FFFFFFF;
            __syncthreads();
            for (int i = 1 + tid; i < M; i += NT)
                if (s_par[i] == n && s_tok[i] == a) atomicMin(&misc->child, i);
            __syncthreads();
            child = (misc->child == 0x7FFFFFFF) ? -1 : misc->child;
        } else if (target_lse) {
            lse_t = target_lse[tb + n];
        }
        if (t1 && !target_lse) {
            // target log-normaliser of row n
            float mx = -__int_as_float(0x7F800000);
            for (int e = tid; e < nch; e += NT) mx = fmaxf(mx, E::val(x[e]));
            mx = dt_warp_max(mx);
            if (lane == 0) misc->red_f[wid] = mx;
            __syncthreads();
            float m_c = misc->red_f[0];
            for (int w = 1; w < NW; ++w) m_c = fmaxf(m_c, misc->red_f[w]);
            __syncthreads();
            float sm = 0.f;
            if (m_c != -__int_as_float(0x7F800000))
                for (int e = tid; e < nch; e += NT) sm += __expf(E::val(x[e]) - m_c);
            sm = dt_warp_sum(sm);
            if (lane == 0) misc->red_f[wid] = sm;
            __syncthreads();
            if (tid == 0) {
                float a = 0.f;
                for (int w = 0; w < NW; ++w) a += misc->red_f[w];
                misc->pub[k & 1].m = m_c;
                misc->pub[k & 1].s = a;
            }
            __syncthreads();
            cluster.sync();
            float pm[SMAX], ps[SMAX];
#pragma unroll
            for (int j = 0; j < SMAX; ++j) {
                pm[j] = -__int_as_float(0x7F800000);
                ps[j] = 0.f;
                if (j < S) {
                    const Pub* r = &cluster.map_shared_rank(misc, j)->pub[k & 1];
                    pm[j] = r->m;
                    ps[j] = r->s;
                }
            }
            float M_ = -__int_as_float(0x7F800000);
#pragma unroll
            for (int j = 0; j < SMAX; ++j) M_ = fmaxf(M_, pm[j]);
            float ssum = 0.f;
#pragma unroll
            for (int j = 0; j < SMAX; ++j)
                if (j < S && pm[j] != -__int_as_float(0x7F800000)) ssum += ps[j] * __expf(pm[j] - M_);
            ++k;
            lse_t = M_ + logf(ssum);
        }
        if (t1) {
            if (c == 0 && tid == 0 && visited_lse) visited_lse[(size_t)b * (L + 1) + len] = lse_t;
            // ratio tests of n's children; the first accepted in rank order wins
            if (tid == 0) { misc->child = 0x7FFFFFFF; misc->nkids = 0; }
            __syncthreads();
            for (int i = 1 + tid; i < M; i += NT) {
                if (s_par[i] != n) continue;
                atomicAdd(&misc->nkids, 1);
                const int tk = s_tok[i];
                const int pos = s_dep[i] - 1;
                const float tv = E::val(trow[tk]);
                const float dv = E::val(draft[((size_t)b * L + pos) * V + tk]);
                const float lpt = __fsub_rn(tv, lse_t);
                const float lpq = __fsub_rn(dv, draft_lse[(size_t)b * L + pos]);
                const float ratio = dt_exp_canon(__fsub_rn(lpt, lpq));
                if (u0[i] < ratio) atomicMin(&misc->child, s_rank[i] * 2048 + i);
            }
            __syncthreads();
            child = (misc->child == 0x7FFFFFFF) ? -1 : (misc->child & 2047);
        }

        if (child >= 0 && len < L) {
            ++len;
            if (c == 0 && tid == 0) acc_nodes[(size_t)b * (L + 1) + len] = child;
            n = child;
            continue;
        }
        if (!t1) break;

        // ---- T=1: draw the replacement / bonus token ------------------------
        const bool has_kids = misc->nkids > 0;
        const int dpos = s_dep[n];  // drafter row of n's children's position
        const T* y = nullptr;
        float lse_d = 0.f;
        if (has_kids) {
            __syncthreads();
            dt_fence_proxy_async();
            unsigned char* dbuf2 = dbuf + (((size_t)chunk * sizeof(T) + 16 + 127) & ~(size_t)127);
            const T* drow = draft + ((size_t)b * L + dpos) * V;
            uint32_t by = 0;
            y = dt_stage_row<T>(drow, lo, hi, dbuf2, &misc->bar, &by);
            if (by) {
                if (tid == 0 && !dt_mbar_wait(&misc->bar, phase)) {
                    misc->timeout = 1;
                    dt_mbar_wait(&misc->bar, phase);
                }
                phase ^= 1;
            }
            lse_d = draft_lse[(size_t)b * L + dpos];
            __syncthreads();
        }
        // two attempts at most: the residual, then P if the residual is empty
        for (int attempt = has_kids ? 0 : 1; attempt < 2; ++attempt) {
            const bool resid = (attempt == 0);
            unsigned long long part = 0;
            for (int e = tid; e < nch; e += NT) {
                unsigned long long P = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(x[e]), lse_t)));
                if (resid) {
                    unsigned long long Q = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(y[e]), lse_d)));
                    P = P > Q ? P - Q : 0ull;
                }
                part += P;
            }
            part = dt_warp_sum_u64(part);
            if (lane == 0) misc->red_u[wid] = part;
            __syncthreads();
            if (tid == 0) {
                unsigned long long a = 0;
                for (int w = 0; w < NW; ++w) a += misc->red_u[w];
                misc->pub[k & 1].u = a;
            }
            __syncthreads();
            cluster.sync();
            unsigned long long sums[SMAX];
#pragma unroll
            for (int j = 0; j < SMAX; ++j) sums[j] = (j < S) ? cluster.map_shared_rank(misc, j)->pub[k & 1].u : 0ull;
            unsigned long long tot = 0, before = 0, mine = 0;
#pragma unroll
            for (int j = 0; j < SMAX; ++j) {
                if (j < c) before += sums[j];
                if (j == c) mine = sums[j];
                tot += sums[j];
            }
            ++k;
            if (tot == 0) continue;  // empty residual: draw from P instead
            float uf = __fmul_rn(u1[n], 16777216.0f);
            unsigned long long X = (unsigned long long)uf;
            if (X > 16777215ull) X = 16777215ull;
            const unsigned long long lo64 = X * tot;
            const unsigned long long hi64 = __umul64hi(X, tot);
            const unsigned long long tgt = (lo64 >> 24) | (hi64 << 40);
            if (tgt >= before && tgt < before + mine) {
                // this CTA holds the draw: scan its chunk in vocabulary order
                const unsigned long long local = tgt - before;
                const int run = (nch + NT - 1) / NT;
                const int e0 = min(nch, tid * run), e1 = min(nch, e0 + run);
                unsigned long long rs = 0;
                for (int e = e0; e < e1; ++e) {
                    unsigned long long P = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(x[e]), lse_t)));
                    if (resid) {
                        unsigned long long Q = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(y[e]), lse_d)));
                        P = P > Q ? P - Q : 0ull;
                    }
                    rs += P;
                }
                // exclusive scan of run sums over the block
                unsigned long long inc = rs;
                for (int o = 1; o < 32; o <<= 1) {
                    unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += t;
                }
                if (lane == 31) misc->scan_u[wid] = inc;
                __syncthreads();
                unsigned long long wb = 0;
                for (int w = 0; w < wid; ++w) wb += misc->scan_u[w];
                const unsigned long long ex = wb + inc - rs;
                if (rs > 0 && local >= ex && local < ex + rs) {
                    unsigned long long acc = ex;
                    for (int e = e0; e < e1; ++e) {
                        unsigned long long P = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(x[e]), lse_t)));
                        if (resid) {
                            unsigned long long Q = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(y[e]), lse_d)));
                            P = P > Q ? P - Q : 0ull;
                        }
                        if (P == 0) continue;
                        acc += P;
                        if (acc > local) { next_tok[b] = lo + e; break; }
                    }
                }
            }
            break;
        }
        break;
    }

    if (c == 0 && tid == 0) {
        acc_len[b] = len;
        if (!t1) next_tok[b] = out_tok;
    }
    if (c == 0)
        for (int i = len + 1 + tid; i <= L; i += NT) acc_nodes[(size_t)b * (L + 1) + i] = -1;
    if (c == 0 && tid == 0) {
        acc_nodes[(size_t)b * (L + 1)] = 0;
        if (visited_lse)
            for (int i = (t1 ? len + 1 : 0); i <= L; ++i) visited_lse[(size_t)b * (L + 1) + i] = 0.f;
    }
    if (tid == 0 && misc->timeout) atomicOr(&status[b], DT_DEV_TIMEOUT);
    __syncthreads();
    cluster.sync();  // keep shared memory alive until every CTA finished its remote reads
}

}  // namespace

size_t dt_kn6_smem_bytes(int chunk, int esize, int Mmax) {
    const size_t tree = (((size_t)Mmax * 16) + 127) & ~(size_t)127;
    const size_t buf = (((size_t)chunk * esize + 16 + 127) & ~(size_t)127);
    return 1024 + tree + 2 * buf;
}

cudaError_t dt_kn6_launch(int batch, int L, int V, int dtype, int Mmax, int S, int chunk, int temperature_one,
                          const int32_t* tok, const int32_t* parent, const int32_t* depth, const int32_t* rank,
                          const int32_t* n_nodes, const float* draft_lse, const void* target,
                          const float* target_lse, const void* draft, const float* uniforms, int32_t* acc_nodes,
                          int32_t* acc_len, int32_t* next_tok, float* visited_lse, int32_t* status,
                          cudaStream_t st) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const size_t smem = dt_kn6_smem_bytes(chunk, esize, Mmax);
    DtLaunch lc(dim3(S, batch, 1), dim3(NT, 1, 1), smem, st, S);
    cudaLaunchConfig_t& cfg = lc.cfg;
    cudaError_t e;
    if (dtype == DT_BF16) {
        auto k = kn6_kernel<uint16_t>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        if (S > 8 && (e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        return cudaLaunchKernelEx(&cfg, k, L, V, Mmax, chunk, temperature_one, tok, parent, depth, rank, n_nodes,
                                  draft_lse, (const uint16_t*)target, target_lse, (const uint16_t*)draft, uniforms,
                                  acc_nodes,
                                  acc_len, next_tok, visited_lse, status);
    } else {
        auto k = kn6_kernel<float>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        if (S > 8 && (e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        return cudaLaunchKernelEx(&cfg, k, L, V, Mmax, chunk, temperature_one, tok, parent, depth, rank, n_nodes,
                                  draft_lse, (const float*)target, target_lse, (const float*)draft, uniforms,
                                  acc_nodes, acc_len,
                                  next_tok, visited_lse, status);
    }
}
