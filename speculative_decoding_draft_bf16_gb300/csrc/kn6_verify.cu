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
// On a tree (the pages give the single-chain rule), three rules at T=1:
//  - ratio (DT_VERIFY_RATIO): at node n the children of n are tested in rank
//    order against p and the walk descends into the first accepted one; if
//    all are rejected the replacement comes from max(0, P - Q) with P, Q the
//    2^32 fixed-point masses of the target row of n and the drafter row of n's
//    children's position (P when the residual is empty); a node without
//    children draws its bonus token from P.
//  - one residual per rejected sibling (DT_VERIFY_ITER_RESIDUAL): child c_1 as
//    above; child c_i (i >= 2) against the residual left by c_1 .. c_{i-1},
//    r_i = [r_{i-1} - q]_+ normalised, held exactly as the integer weights
//    W_i = max(0, P - floor(Q * T_i / 2^32)), T_1 = 2^32, T_{i+1} = T_i + sum W_i
//    (one pass over the row per rejected child); the replacement comes from
//    the last residual.
//  - exact target-sample matching (DT_VERIFY_TARGET_MATCH, as DFlash does per
//    [DARTree] "Speculative sampling"): at every node draw from P and descend
//    while the draw is a child's token; the drafter rows are not read.
// Ratios and masses use dt_exp_canon, and the draws are exact integer inverse
// CDFs, so results are reproducible.
//
// One thread-block cluster of S CTAs per request; CTA c owns a vocabulary
// chunk.  Rows are bulk-copied chunk-wise into shared memory: the target row
// of each visited node (at T=1 with caller-supplied normalisers only the last
// one) and, at T=1, the drafter row of the children's position of each
// visited inner node (for the residual).  While node n is processed, the
// target row of n's rank-0 child (the drafter's favourite, the likeliest next
// node) is already on its way into a second buffer, so an accepted favourite
// costs no copy latency.  Partial argmax / (max, sum exp) / residual sums are
// combined across the cluster through distributed shared memory.  The
// residual draw computes each thread's run of masses once; the CTA holding the
// draw scans the run sums, and one warp re-walks the single run that holds it.
#include "dt_device.cuh"
#include "dt_exp.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int SMAX = 16;
constexpr int NBMAX = 3;  // row buffers: up to two target rows, one drafter row

struct Pub {
    float m, s;
    unsigned long long u, w;
};

struct Kn6Misc {
    uint64_t bar[NBMAX];
    uint64_t probe;               // the timeout-path test hook's barrier (never completes)
    int timeout;
    int bad;
    Pub pub[2];
    unsigned long long red_u[NW];
    unsigned long long red_w[NW];
    float red_f[NW];
    int child;
    int drawn[2];                 // matching: the token drawn by the CTA holding the draw
    unsigned long long best_kid;
    float xm[SMAX];               // partners' published values, copied through DSMEM
    float xs[SMAX];
    unsigned long long xu[SMAX];  // greedy: partners' argmax keys
    // residual and mass sums of every CTA of the cluster, pushed by each into
    // slot c of every CTA before a cluster barrier; two buffers by exchange parity
    unsigned long long su[2][SMAX];
    unsigned long long sw[2][SMAX];
    int nkid;                     // children of the node whose residual loop runs
    int scan[NW];                 // per-warp totals of a block scan
};
constexpr size_t MISC_BYTES = 2048;
static_assert(sizeof(Kn6Misc) <= MISC_BYTES, "misc block overflows its slot");

DT_DI unsigned long long warp_max_u64(unsigned long long v) {
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long t = __shfl_xor_sync(0xffffffffu, v, o);
        v = t > v ? t : v;
    }
    return v;
}

DT_DI unsigned long long warp_incl_scan_u64(unsigned long long v) {
    const int lane = threadIdx.x & 31;
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Residual weight max(0, P - floor(Q * T / 2^32)) (Q <= 2^32, T < 2^44).
DT_DI unsigned long long resid_w(unsigned long long P, unsigned long long Q, unsigned long long T) {
    const unsigned long long s = ((Q * T) >> 32) | (__umul64hi(Q, T) << 32);
    return P > s ? P - s : 0ull;
}
// The same for 32-bit P and Q (Q < 2^32), T split as Th * 2^32 + Tl:
// floor(Q * T / 2^32) = Q * Th + floor(Q * Tl / 2^32), two 32 x 32 -> 64-bit products.
DT_DI unsigned long long resid_w32(uint32_t P, uint32_t Q, uint32_t Th, uint32_t Tl) {
    const unsigned long long s = (unsigned long long)Q * Th + (((unsigned long long)Q * Tl) >> 32);
    return (unsigned long long)P > s ? (unsigned long long)P - s : 0ull;
}

// Test of a child against the residual with weights W (sum S):
// floor(u * 2^24) * Q * S < W * 2^56, in 128-bit integers.
DT_DI bool resid_accepts(float u, unsigned long long Q, unsigned long long S, unsigned long long W) {
    unsigned long long X = (unsigned long long)__fmul_rn(u, 16777216.0f);
    if (X > 16777215ull) X = 16777215ull;
    const unsigned long long a = X * Q;
    const unsigned long long lhi = __umul64hi(a, S), llo = a * S;
    const unsigned long long rhi = W >> 8, rlo = W << 56;
    return lhi < rhi || (lhi == rhi && llo < rlo);
}

// 2^32 fixed-point probability mass exp(v - lse) of one element, or its
// residual weight resid_w(P, Q, T) when resid.
DT_DI unsigned long long mass(float xv, float lse_t, bool resid, float yv, float lse_d, unsigned long long T) {
    const unsigned long long P = dt_fixed32(dt_exp_canon(__fsub_rn(xv, lse_t)));
    if (!resid) return P;
    return resid_w(P, dt_fixed32(dt_exp_canon(__fsub_rn(yv, lse_d))), T);
}

// Row buffers of one CTA.  Every thread keeps an identical copy of this state
// (named scalars and bit masks rather than arrays, so it stays in registers).
template <typename T>
struct Rows {
    unsigned char* base;  // buffer 0; buffer i at base + i * stride
    int stride;
    uint64_t* bar;
    int h0, h1, h2;       // head misalignment (elements) of the chunk staged in each buffer
    int t0, t1, t2;       // which row (target: node, drafter: position) a buffer holds; -1 none
    uint32_t pend;        // bit i: a bulk copy into buffer i has not been waited for
    uint32_t ph;          // bit i: mbarrier phase parity of buffer i
    DtStager<T> s0, s1, s2;  // ragged chunk ends of each buffer's latest copy, in registers
    uint64_t* probe;      // the timeout-path test hook's barrier, and its budget (0: off)
    long long probe_budget;

    DT_DI void init(unsigned char* b, int s, uint64_t* bars, uint64_t* probe_bar, long long pb) {
        base = b;
        stride = s;
        bar = bars;
        probe = probe_bar;
        probe_budget = pb;
        h0 = h1 = h2 = 0;
        t0 = t1 = t2 = -1;
        pend = ph = 0;
        s0.held_off = s1.held_off = s2.held_off = -1;
    }
    DT_DI int holds(int i) const { return i == 0 ? t0 : (i == 1 ? t1 : t2); }
    DT_DI int head(int i) const { return i == 0 ? h0 : (i == 1 ? h1 : h2); }
    DT_DI const uint4* vec(int i) const { return (const uint4*)(base + (size_t)i * stride); }
    DT_DI const T* elems(int i) const { return (const T*)(base + (size_t)i * stride) + head(i); }
    // Completes buffer i: stores its ragged ends, then one thread waits for
    // its bulk copy.  The caller syncs the block before reading.
    DT_DI void wait(int i, int* timeout) {
        unsigned char* dst = base + (size_t)i * stride;
        if (i == 0) s0.finish(dst);
        else if (i == 1) s1.finish(dst);
        else s2.finish(dst);
        if (i == 0) s0.held_off = -1;
        else if (i == 1) s1.held_off = -1;
        else s2.held_off = -1;
        if (!((pend >> i) & 1u)) return;
        if (threadIdx.x == 0 && !dt_probe_wait(probe, probe_budget)) *timeout = 1;
        if (threadIdx.x == 0 && !dt_mbar_wait(&bar[i], (ph >> i) & 1u)) {
            *timeout = 1;
            dt_mbar_wait(&bar[i], (ph >> i) & 1u);
        }
        ph ^= 1u << i;
        pend &= ~(1u << i);
    }
    // Starts copying chunk [lo, hi) of `row` into buffer i (all threads).  Any
    // earlier copy into it is waited for first, and all earlier reads of it
    // are ordered before the new writes.
    DT_DI void stage(int i, const T* row, int tag, int lo, int hi, int* timeout) {
        wait(i, timeout);
        __syncthreads();
        dt_fence_proxy_async();
        unsigned char* dst = base + (size_t)i * stride;
        const uint32_t bytes = i == 0 ? s0.start(row, lo, hi, dst, &bar[i])
                                      : (i == 1 ? s1.start(row, lo, hi, dst, &bar[i]) : s2.start(row, lo, hi, dst, &bar[i]));
        const int hd = (int)(((uintptr_t)(row + lo) & 15u) / sizeof(T));
        if (bytes) pend |= 1u << i;
        if (i == 0) { h0 = hd; t0 = tag; }
        else if (i == 1) { h1 = hd; t1 = tag; }
        else { h2 = hd; t2 = tag; }
    }
};

// The normalised DARTree proposal q~(v | u) = exp(((d[v] - lse) + <U[u], Vt[v]>) - z)
// of a node's children (u: the node's token, z: its log-normaliser row).
struct Kn6Corr {
    const float* U;         // [V][R] fp32
    const float* Vt;        // [V][R] fp32, 16-byte aligned, R % 4 == 0
    int R;                  // <= 64
    const float* z;         // [batch][L][K] log-normalisers
    int K;
    const int32_t* root_tok;  // [batch] or NULL
};

// Probe budget of the timeout-path test hook (0: off), set by dt_kn6_set_probe.
__device__ long long g_kn6_probe;

// One instantiation per acceptance rule (RULE = DT_VERIFY_*), so that each
// walk carries only its own code; CORR: the ratio rule against q~.
template <typename T, int RULE, bool CORR>
__global__ void __launch_bounds__(NT, 2) kn6_kernel(Kn6Corr corr, int L, int V, int Mmax, int chunk, int nbt, int pq_cap,
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
    constexpr int EPV = 16 / sizeof(T);
    __shared__ __align__(16) float s_ur[CORR ? 64 : 4];  // U row of the proposing node's token
    const float NEG_INF = -__int_as_float(0x7F800000);
    extern __shared__ __align__(128) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int c = (int)cluster.block_rank();
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int lo = min(V, c * chunk), hi = min(V, lo + chunk);
    const int nch = hi - lo;

    Kn6Misc* misc = (Kn6Misc*)smem;
    int* s_tok = (int*)(smem + MISC_BYTES);
    int* s_par = s_tok + Mmax;
    int* s_dep = s_par + Mmax;
    int* s_rank = s_dep + Mmax;
    int* s_nk = s_rank + Mmax;    // children per node
    int* s_pred = s_nk + Mmax;    // rank-0 child (smallest index), INT_MAX if none
    const size_t tree_bytes = ((size_t)Mmax * 24 + 127) & ~(size_t)127;
    const int DB = nbt;           // index of the drafter buffer

    Rows<T> rows;
    // the residual-per-sibling rule keeps its ordered children before the row
    // buffers, so that its pair cache may take the buffers' place
    const size_t kids_bytes = RULE == DT_VERIFY_ITER_RESIDUAL ? (((size_t)Mmax * 24) + 127) & ~(size_t)127 : 0;
    rows.init(smem + MISC_BYTES + tree_bytes + kids_bytes,
              (int)(((size_t)chunk * sizeof(T) + 16 + 127) & ~(size_t)127), misc->bar, &misc->probe, g_kn6_probe);

    if (tid == 0) {
        for (int i = 0; i < NBMAX; ++i) dt_mbar_init(&misc->bar[i], 1);
        dt_mbar_init(&misc->probe, 1);
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
            s_nk[i] = 0;
            s_pred[i] = 0x7FFFFFFF;
        }
        __syncthreads();
        for (int i = tid; i < M; i += NT) {
            const int p = s_par[i], d = s_dep[i];
            bool ok;
            if (i == 0) ok = (p == -1 && d == 0);
            else ok = (p >= 0 && p < M && p != i && d >= 1 && d <= L && d == s_dep[p] + 1 && s_tok[i] >= 0 &&
                       s_tok[i] < V);
            if (!ok) misc->bad = 1;
            else if (i > 0) {
                atomicAdd(&s_nk[p], 1);
                if (s_rank[i] == 0) atomicMin(&s_pred[p], i);
            }
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
    int cur = 0;  // target buffer holding row n
    int k = 0;    // cluster exchanges so far (selects the Pub slot)
    int out_tok = -1;
    constexpr int rule = RULE;
    constexpr bool greedy = rule == DT_VERIFY_GREEDY;
    constexpr bool match = rule == DT_VERIFY_TARGET_MATCH;
    constexpr bool uses_q = rule == DT_VERIFY_RATIO || rule == DT_VERIFY_ITER_RESIDUAL;
    const float* u0 = uniforms ? uniforms + (size_t)b * 2 * Mmax : nullptr;
    const float* u1 = u0 ? u0 + Mmax : nullptr;
    // per-node target rows: argmax (T=0), a draw at every node (matching), or
    // the normaliser (T=1 without target_lse)
    const bool rows_needed = greedy || match || !target_lse;
    auto trow_of = [&](int node) { return target + (tb + node) * (size_t)V; };
    auto drow_of = [&](int pos) { return draft + ((size_t)b * L + pos) * V; };
    // children are tested in (rank, index) order
    auto kid_key = [&](int i) {
        return ((unsigned long long)((uint32_t)s_rank[i] ^ 0x80000000u) << 32) | (uint32_t)i;
    };
    // accept `ch` as the next path node
    auto descend = [&](int ch) {
        ++len;
        if (c == 0 && tid == 0) acc_nodes[(size_t)b * (L + 1) + len] = ch;
        n = ch;
        if (rows_needed) {
            if (nbt == 2 && rows.holds(cur ^ 1) == ch) cur ^= 1;
            else rows.stage(cur, trow_of(ch), ch, lo, hi, &misc->timeout);
        }
    };
    if (rows_needed) rows.stage(cur, trow_of(0), 0, lo, hi, &misc->timeout);

    for (;;) {
        // ---- copies for what may come next -----------------------------------
        const int pred = s_pred[n];
        if (rows_needed && nbt == 2 && pred != 0x7FFFFFFF && len < L && rows.holds(cur ^ 1) != pred)
            rows.stage(cur ^ 1, trow_of(pred), pred, lo, hi, &misc->timeout);
        if (uses_q && s_nk[n] > 0 && rows.holds(DB) != s_dep[n])
            rows.stage(DB, drow_of(s_dep[n]), s_dep[n], lo, hi, &misc->timeout);

        int child = -1;
        float lse_t = 0.f;
        const uint4* xv = rows.vec(cur);
        const int h = rows.head(cur);
        const int nv = (h + nch + EPV - 1) / EPV;
        const int full_lo = (h > 0) ? 1 : 0;
        const int full_hi = ((h + nch) % EPV == 0) ? nv : nv - 1;
        if (rows_needed) {
            rows.wait(cur, &misc->timeout);
            __syncthreads();
        }
        if (greedy) {
            // argmax, smallest id on ties: each thread keeps the first of its
            // vectors holding its largest value, then the first such element
            float lb = NEG_INF;
            int lj = -1;
            for (int j = tid; j < nv; j += NT) {
                const uint4 q = xv[j];
                float vm;
                if (j >= full_lo && j < full_hi) {
                    vm = dt_vec_max<T>(q);
                } else {
                    float xe[EPV];
                    dt_vec_vals<T>(q, xe);
                    vm = NEG_INF;
#pragma unroll
                    for (int s = 0; s < EPV; ++s) {
                        const int idx = j * EPV + s - h;
                        if (idx >= 0 && idx < nch) vm = fmaxf(vm, xe[s]);
                    }
                }
                if (vm > lb || lj < 0) { lb = vm; lj = j; }
            }
            unsigned long long best = 0;
            if (lj >= 0) {
                float xe[EPV];
                dt_vec_vals<T>(xv[lj], xe);
                int id = -1;
#pragma unroll
                for (int s = EPV - 1; s >= 0; --s) {
                    const int idx = lj * EPV + s - h;
                    if (idx >= 0 && idx < nch && xe[s] == lb) id = lo + idx;
                }
                best = ((unsigned long long)E::key(dt_to_elem<T>(lb)) << 32) |
                       (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
            }
            best = warp_max_u64(best);
            if (lane == 0) misc->red_u[wid] = best;
            __syncthreads();
            if (tid == 0) {
                unsigned long long a = 0;
                for (int w = 0; w < NW; ++w) a = misc->red_u[w] > a ? misc->red_u[w] : a;
                misc->pub[k & 1].u = a;
                misc->child = 0x7FFFFFFF;
            }
            __syncthreads();
            cluster.sync();
            if (tid < S) misc->xu[tid] = cluster.map_shared_rank(misc, tid)->pub[k & 1].u;
            __syncthreads();
            unsigned long long g = 0;
            for (int j = 0; j < S; ++j) g = misc->xu[j] > g ? misc->xu[j] : g;
            ++k;
            const int a = (int)(0xFFFFFFFFu - (uint32_t)(g & 0xFFFFFFFFull));
            out_tok = a;
            if (s_nk[n] > 0)
                for (int i = 1 + tid; i < M; i += NT)
                    if (s_par[i] == n && s_tok[i] == a) atomicMin(&misc->child, i);
            __syncthreads();
            child = (misc->child == 0x7FFFFFFF) ? -1 : misc->child;
        } else if (target_lse) {
            lse_t = target_lse[tb + n];
        } else {
            // target log-normaliser of row n: chunk max, then sum exp(x - max)
            float lm = NEG_INF;
            for (int j = tid; j < nv; j += NT) {
                const uint4 q = xv[j];
                if (j >= full_lo && j < full_hi) {
                    lm = fmaxf(lm, dt_vec_max<T>(q));
                } else {
                    float xe[EPV];
                    dt_vec_vals<T>(q, xe);
#pragma unroll
                    for (int s = 0; s < EPV; ++s) {
                        const int idx = j * EPV + s - h;
                        if (idx >= 0 && idx < nch) lm = fmaxf(lm, xe[s]);
                    }
                }
            }
            lm = dt_warp_max(lm);
            if (lane == 0) misc->red_f[wid] = lm;
            __syncthreads();
            float m_c = NEG_INF;
#pragma unroll
            for (int w = 0; w < NW; ++w) m_c = fmaxf(m_c, misc->red_f[w]);
            const float log2e = 1.44269504088896340736f;
            float sm = 0.f;
            if (m_c != NEG_INF) {
                const unsigned long long m2 = dt_f2_pack(m_c, m_c), l2 = dt_f2_pack(log2e, log2e);
                unsigned long long acc = dt_f2_pack(0.f, 0.f);
                for (int j = tid; j < nv; j += NT) {
                    const uint4 q = xv[j];
                    if (j >= full_lo && j < full_hi) {
                        acc = dt_vec_expsum<T>(q, m2, l2, acc);
                    } else {
                        float xe[EPV];
                        dt_vec_vals<T>(q, xe);
#pragma unroll
                        for (int s = 0; s < EPV; ++s) {
                            const int idx = j * EPV + s - h;
                            if (idx >= 0 && idx < nch) sm += dt_ex2_approx(__fmul_rn(__fsub_rn(xe[s], m_c), log2e));
                        }
                    }
                }
                float a0, a1;
                dt_f2_unpack(acc, a0, a1);
                sm += a0 + a1;
            }
            sm = dt_warp_sum(sm);
            __syncthreads();  // every thread has read red_f
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
            if (tid < S) {
                const Pub* r = &cluster.map_shared_rank(misc, tid)->pub[k & 1];
                misc->xm[tid] = r->m;
                misc->xs[tid] = r->s;
            }
            __syncthreads();
            float M_ = NEG_INF;
            for (int j = 0; j < S; ++j) M_ = fmaxf(M_, misc->xm[j]);
            float ssum = 0.f;
            for (int j = 0; j < S; ++j)
                if (misc->xm[j] != NEG_INF) ssum += misc->xs[j] * __expf(misc->xm[j] - M_);
            ++k;
            lse_t = M_ + logf(ssum);
        }
        // the proposal of n's children: q~ needs n's token (the root: root_tok)
        // and log-normaliser, and the U row staged for the dot products
        int qu = -1;
        float qz = 0.f;
        if constexpr (CORR) {
            qu = n == 0 ? (corr.root_tok ? corr.root_tok[b] : -1) : s_tok[n];
            if (qu >= V || s_dep[n] >= L) qu = -1;
            if (qu >= 0) {
                qz = corr.z[((size_t)b * L + s_dep[n]) * corr.K + (n == 0 ? 0 : s_rank[n])];
                if (tid < corr.R) s_ur[tid] = corr.U[(size_t)qu * corr.R + tid];
            }
            __syncthreads();
        }
        // <U[qu], Vt[v]>: serial fp32 fma from 0 over the R columns
        auto markov_dot = [&](int v) {
            float acc = 0.f;
            const float4* vr = (const float4*)(corr.Vt + (size_t)v * corr.R);
            for (int k4 = 0; k4 < (corr.R >> 2); ++k4) {
                const float4 q = vr[k4];
                acc = __fmaf_rn(s_ur[4 * k4 + 0], q.x, acc);
                acc = __fmaf_rn(s_ur[4 * k4 + 1], q.y, acc);
                acc = __fmaf_rn(s_ur[4 * k4 + 2], q.z, acc);
                acc = __fmaf_rn(s_ur[4 * k4 + 3], q.w, acc);
            }
            return acc;
        };
        // log q of token v at n's children's position from its drafter value dv
        auto proposal_lp = [&](float dv, float dlse, int v) {
            float l = __fsub_rn(dv, dlse);
            if constexpr (CORR) {
                if (qu >= 0) {
                    l = __fadd_rn(l, markov_dot(v));
                    l = __fsub_rn(l, qz);
                }
            }
            return l;
        };
        // single-residual test of child i against p (fp32, exp_canon ratio)
        auto ratio_accepts = [&](int i) {
            const int tk = s_tok[i];
            const int pos = s_dep[i] - 1;
            const float tv = E::val(trow_of(n)[tk]);
            const float dv = E::val(drow_of(pos)[tk]);
            const float lpt = __fsub_rn(tv, lse_t);
            const float lpq = proposal_lp(dv, draft_lse[(size_t)b * L + pos], tk);
            return u0[i] < dt_exp_canon(__fsub_rn(lpt, lpq));
        };
        if (!greedy) {
            if (c == 0 && tid == 0 && visited_lse) visited_lse[(size_t)b * (L + 1) + len] = lse_t;
            if (uses_q) {
                // ratio rule: every child against p, the first accepted in (rank, index)
                // order wins; residual rule: find the first child and test it alone
                if (tid == 0) misc->best_kid = ~0ull;
                __syncthreads();
                if (s_nk[n] > 0) {
                    for (int i = 1 + tid; i < M; i += NT) {
                        if (s_par[i] != n) continue;
                        if (rule != DT_VERIFY_RATIO || ratio_accepts(i)) atomicMin(&misc->best_kid, kid_key(i));
                    }
                }
                __syncthreads();
                const unsigned long long bk = misc->best_kid;
                if (rule == DT_VERIFY_RATIO) {
                    child = (bk == ~0ull) ? -1 : (int)(bk & 0xFFFFFFFFull);
                } else if (bk != ~0ull) {  // the first child in test order
                    if (ratio_accepts((int)(bk & 0xFFFFFFFFull))) child = (int)(bk & 0xFFFFFFFFull);
                }
            }
        }

        if (child >= 0 && len < L) {
            descend(child);
            continue;
        }
        if (greedy) break;

        // ---- T=1: residuals and the draw -------------------------------------
        const bool has_kids = s_nk[n] > 0;
        const bool resid = uses_q && has_kids;
        if (rows.holds(cur) != n) rows.stage(cur, trow_of(n), n, lo, hi, &misc->timeout);
        rows.wait(cur, &misc->timeout);
        float lse_d = 0.f;
        if (resid) {
            rows.wait(DB, &misc->timeout);
            lse_d = draft_lse[(size_t)b * L + s_dep[n]];
        }
        __syncthreads();
        const T* x = rows.elems(cur);
        const T* y = rows.elems(DB);
        // masses of a contiguous run of elements per thread (odd length, so
        // that the lanes' 2- or 4-byte reads spread over the banks)
        const int run = ((nch + NT - 1) / NT) | 1;
        const int e0 = min(nch, tid * run), e1 = min(nch, e0 + run);
        unsigned long long Tq = 1ull << 32;  // residual weights max(0, P - floor(Q * Tq / 2^32))
        unsigned long long rR = 0, rP = 0, totR = 0;
        // one residual per sibling: the CTA keeps the (P, Q) pairs whose weight
        // is still positive, 32 bits each, every thread its own in a segment
        // of pq (sized by a scan of the threads' counts), and drops a pair once
        // its weight reaches 0 (weights only fall as T grows).  The cache takes
        // the place of the staged rows, which from then on are read from
        // global memory (the fill, a recompute, the draw).  When the pairs do
        // not fit (pq_cap pairs), or the CTA holds a 2^32 mass (a one-hot row),
        // every step recomputes the runs instead.
        const bool iter = rule == DT_VERIFY_ITER_RESIDUAL && resid;
        uint2* pq = (uint2*)(smem + MISC_BYTES + tree_bytes + kids_bytes);  // over the row buffers
        int na = 0;
        bool sat = false;
        for (int e = e0; e < e1; ++e) {
            const unsigned long long P = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(x[e]), lse_t)));
            rP += P;
            if (resid) {
                const unsigned long long Q = dt_fixed32(dt_exp_canon(proposal_lp(E::val(y[e]), lse_d, lo + e)));
                const unsigned long long w = P > Q ? P - Q : 0ull;
                rR += w;
                if (iter && w) {
                    sat |= ((P | Q) >> 32) != 0;
                    na += Q != 0;  // Q = 0: the weight stays P at every T (summed once, below)
                }
            }
        }
        bool use_pq = false;
        int seg = 0;                   // this thread's first pair in pq
        unsigned long long rconst = 0;  // cached mode: the weights of the run's Q = 0 elements
        if (iter && pq_cap > 0 && !__syncthreads_or(sat)) {
            // exclusive scan of the pair counts; cache only if the CTA's fit
            const int inc = dt_warp_incl_scan(na);
            if (lane == 31) misc->scan[wid] = inc;
            __syncthreads();
            int before = 0, total = 0;
            for (int w = 0; w < NW; ++w) {
                if (w < wid) before += misc->scan[w];
                total += misc->scan[w];
            }
            seg = before + inc - na;
            use_pq = total <= pq_cap;
            __syncthreads();  // every thread has read scan and is done with the staged rows
            if (use_pq) {
                x = trow_of(n) + lo;  // the rows again, from global memory
                y = drow_of(s_dep[n]) + lo;
                int j = seg;
                for (int e = e0; e < e1; ++e) {
                    const unsigned long long P = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(x[e]), lse_t)));
                    const unsigned long long Q = dt_fixed32(dt_exp_canon(proposal_lp(E::val(y[e]), lse_d, lo + e)));
                    if (P > Q) {
                        if (Q) pq[j++] = make_uint2((uint32_t)P, (uint32_t)Q);
                        else rconst += P;
                    }
                }
                __syncthreads();
            }
        }
        // the node's children in test order (rank, then index), with the masses
        // and uniforms of their tests, once per node
        unsigned long long* kidP = (unsigned long long*)(smem + MISC_BYTES + tree_bytes);
        unsigned long long* kidQ = kidP + Mmax;
        int* kidI = (int*)(kidQ + Mmax);
        float* kidU = (float*)(kidI + Mmax);
        int nk = 0;
        if (iter) {
            int* unord = (int*)kidQ;  // the children gathered in any order (kidQ is filled after)
            if (tid == 0) misc->nkid = 0;
            __syncthreads();
            for (int i = 1 + tid; i < M; i += NT)
                if (s_par[i] == n) unord[atomicAdd(&misc->nkid, 1)] = i;
            __syncthreads();
            nk = misc->nkid;
            for (int q = tid; q < nk; q += NT) {
                const int i = unord[q];
                const unsigned long long ki = kid_key(i);
                int pos = 0;
                for (int r = 0; r < nk; ++r) pos += kid_key(unord[r]) < ki;
                kidI[pos] = i;
            }
            __syncthreads();  // the order is complete and the gathered list no longer read
            const float dl = draft_lse[(size_t)b * L + s_dep[n]];
            for (int q = tid; q < nk; q += NT) {
                const int i = kidI[q], tk = s_tok[i];
                kidP[q] = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(trow_of(n)[tk]), lse_t)));
                kidQ[q] = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(drow_of(s_dep[n])[tk]), dl)));
                kidU[q] = u0[i];
            }
            __syncthreads();
        }
        // cluster-wide sums of the threads' run sums: each CTA pushes its sum
        // into slot c of every CTA (parity k & 1), one barrier, local adds
        auto cluster_sum = [&](unsigned long long v, unsigned long long w, bool with_w) {
            const unsigned long long sv = dt_warp_sum_u64(v), sw = with_w ? dt_warp_sum_u64(w) : 0ull;
            if (lane == 0) {
                misc->red_u[wid] = sv;
                misc->red_w[wid] = sw;
            }
            __syncthreads();
            if (wid == 0) {
                unsigned long long av = lane < NW ? misc->red_u[lane] : 0ull;
                unsigned long long aw = (with_w && lane < NW) ? misc->red_w[lane] : 0ull;
                av = dt_warp_sum_u64(av);
                aw = dt_warp_sum_u64(aw);
                if (lane < S) {
                    Kn6Misc* r = cluster.map_shared_rank(misc, lane);
                    r->su[k & 1][c] = av;
                    if (with_w) r->sw[k & 1][c] = aw;
                }
            }
            cluster.sync();
            ++k;
        };
        child = -1;
        int kpos = 1;  // the first child was tested against p above
        const unsigned long long* swp = nullptr;  // the CTAs' P sums (first exchange)
        for (bool first = true;; first = false) {
            if (!first) {  // a later residual: T has grown
                rR = 0;
                if (use_pq) {
                    // four pairs per step (independent loads and products); the
                    // survivors are written back in order to the segment's front
                    const uint32_t Th = (uint32_t)(Tq >> 32), Tl = (uint32_t)Tq;
                    rR = rconst;
                    int keep = 0, j = 0;
                    for (; j + 4 <= na; j += 4) {
                        const uint2 v0 = pq[seg + j], v1 = pq[seg + j + 1], v2 = pq[seg + j + 2], v3 = pq[seg + j + 3];
                        const unsigned long long w0 = resid_w32(v0.x, v0.y, Th, Tl), w1 = resid_w32(v1.x, v1.y, Th, Tl);
                        const unsigned long long w2 = resid_w32(v2.x, v2.y, Th, Tl), w3 = resid_w32(v3.x, v3.y, Th, Tl);
                        rR += (w0 + w1) + (w2 + w3);
                        if (w0) pq[seg + keep++] = v0;
                        if (w1) pq[seg + keep++] = v1;
                        if (w2) pq[seg + keep++] = v2;
                        if (w3) pq[seg + keep++] = v3;
                    }
                    for (; j < na; ++j) {
                        const uint2 v = pq[seg + j];
                        const unsigned long long w = resid_w32(v.x, v.y, Th, Tl);
                        rR += w;
                        if (w) pq[seg + keep++] = v;
                    }
                    na = keep;
                } else {
                    for (int e = e0; e < e1; ++e)
                        rR += mass(E::val(x[e]), lse_t, true, E::val(y[e]), lse_d, Tq);
                }
            }
            cluster_sum(rR, rP, first);
            const unsigned long long* su = misc->su[(k - 1) & 1];
            if (first) swp = misc->sw[(k - 1) & 1];
            totR = dt_warp_sum_u64(lane < S ? su[lane] : 0ull);  // the S partials, loaded in parallel
            if (!iter || totR == 0 || kpos >= nk) break;
            // the next child in test order, against the residual just summed
            // (every thread takes the same decision from the same values)
            if (resid_accepts(kidU[kpos], kidQ[kpos], totR, resid_w(kidP[kpos], kidQ[kpos], Tq))) {
                child = kidI[kpos];
                break;
            }
            ++kpos;
            Tq += totR;
        }
        if (child >= 0) {
            descend(child);
            continue;
        }

        // the residual, or P where the residual is empty (or the node has no
        // children, or the rule draws from the target)
        const bool use_r = resid && totR > 0;
        const unsigned long long* sums = use_r ? misc->su[(k - 1) & 1] : swp;
        unsigned long long tot = 0, before = 0, mine = 0;
        for (int j = 0; j < S; ++j) {
            const unsigned long long v = sums[j];
            if (j < c) before += v;
            if (j == c) mine = v;
            tot += v;
        }
        // matching at an inner node: the draw decides the next node, so every
        // CTA needs it; elsewhere it is the emitted token
        const bool bcast = match && has_kids && len < L;
        if (tid == 0) misc->drawn[k & 1] = -1;  // ordered before the holder's write by its barriers
        int holder = -1;
        if (tot > 0) {
            float uf = __fmul_rn(u1[n], 16777216.0f);
            unsigned long long X = (unsigned long long)uf;
            if (X > 16777215ull) X = 16777215ull;
            const unsigned long long lo64 = X * tot;
            const unsigned long long hi64 = __umul64hi(X, tot);
            const unsigned long long tgt = (lo64 >> 24) | (hi64 << 40);
            unsigned long long cum = 0;
            for (int j = 0; j < S; ++j) {
                if (holder < 0 && tgt >= cum && tgt < cum + sums[j]) holder = j;
                cum += sums[j];
            }
            if (holder == c) {
                // this CTA holds the draw: exclusive scan of the run sums
                const unsigned long long rs = use_r ? rR : rP;
                const unsigned long long inc = warp_incl_scan_u64(rs);
                __syncthreads();  // red_u was read by tid 0 above
                if (lane == 31) misc->red_u[wid] = inc;
                __syncthreads();
                unsigned long long wb = 0;
                for (int w = 0; w < wid; ++w) wb += misc->red_u[w];
                const unsigned long long ex = wb + inc - rs;
                const unsigned long long local = tgt - before;
                const bool hit = rs > 0 && local >= ex && local < ex + rs;
                const unsigned hm = __ballot_sync(0xffffffffu, hit);
                if (hm) {
                    // one warp re-walks the run that holds the draw, 32 elements at a time
                    const int src = __ffs(hm) - 1;
                    const int a0 = __shfl_sync(0xffffffffu, e0, src), a1 = __shfl_sync(0xffffffffu, e1, src);
                    unsigned long long base = __shfl_sync(0xffffffffu, ex, src);
                    for (int g0 = a0; g0 < a1; g0 += 32) {
                        const int e = g0 + lane;
                        unsigned long long P = 0;
                        if (e < a1) {
                            P = dt_fixed32(dt_exp_canon(__fsub_rn(E::val(x[e]), lse_t)));
                            if (use_r)
                                P = resid_w(P, dt_fixed32(dt_exp_canon(proposal_lp(E::val(y[e]), lse_d, lo + e))), Tq);
                        }
                        const unsigned long long ci = warp_incl_scan_u64(P);
                        const unsigned found = __ballot_sync(0xffffffffu, P > 0 && base + ci > local);
                        if (found) {
                            if (lane == __ffs(found) - 1) {
                                if (bcast) misc->drawn[k & 1] = lo + e;
                                else next_tok[b] = lo + e;
                            }
                            break;
                        }
                        base += __shfl_sync(0xffffffffu, ci, 31);
                    }
                }
            }
        } else if (c == 0 && tid == 0) {
            next_tok[b] = -1;  // no mass to draw from
        }
        if (bcast && tot > 0) {
            __syncthreads();
            cluster.sync();
            if (tid == 0) misc->child = cluster.map_shared_rank(misc, holder)->drawn[k & 1];
            __syncthreads();
            const int yt = misc->child;
            ++k;
            __syncthreads();  // every thread has read misc->child
            if (tid == 0) misc->child = 0x7FFFFFFF;
            __syncthreads();
            for (int i = 1 + tid; i < M; i += NT)
                if (s_par[i] == n && s_tok[i] == yt) atomicMin(&misc->child, i);
            __syncthreads();
            const int ch = misc->child;
            if (ch != 0x7FFFFFFF) {
                descend(ch);
                continue;
            }
            if (c == 0 && tid == 0) next_tok[b] = yt;
        }
        break;
    }

    if (c == 0 && tid == 0) {
        acc_len[b] = len;
        if (greedy) next_tok[b] = out_tok;
    }
    if (c == 0)
        for (int i = len + 1 + tid; i <= L; i += NT) acc_nodes[(size_t)b * (L + 1) + i] = -1;
    if (c == 0 && tid == 0) {
        acc_nodes[(size_t)b * (L + 1)] = 0;
        if (visited_lse)
            for (int i = (greedy ? 0 : len + 1); i <= L; ++i) visited_lse[(size_t)b * (L + 1) + i] = 0.f;
    }
    // no copy may still be landing in shared memory when the CTA exits
#pragma unroll
    for (int i = 0; i < NBMAX; ++i) rows.wait(i, &misc->timeout);
    __syncthreads();
    if (tid == 0 && misc->timeout) atomicOr(&status[b], DT_DEV_TIMEOUT);
    cluster.sync();  // keep shared memory alive until every CTA finished its remote reads
}

// Shared-memory layout: misc (2 KB), tree, nbt target-row buffers and one
// drafter-row buffer.  For the residual-per-sibling rule: misc, tree, the
// ordered children of a node with their test values (24 bytes per node), one
// target-row and one drafter-row buffer, and over those buffers a cache of
// `cap` (P, Q) pairs (8 bytes each) for the CTA's alive elements, up to the
// chunk, within the shared memory.  Two target buffers (prefetch of the
// favourite child) when they fit, for the other rules.
struct Kn6Layout {
    int nbt, cap;
    size_t total;
};
Kn6Layout kn6_layout(int chunk, int esize, int Mmax, int rule) {
    const size_t tree = (((size_t)Mmax * 24) + 127) & ~(size_t)127;
    const size_t buf = (((size_t)chunk * esize + 16 + 127) & ~(size_t)127);
    const size_t room = (size_t)226 * 1024;
    auto base = [&](int nbt) { return MISC_BYTES + tree + (size_t)(nbt + 1) * buf; };
    if (rule != DT_VERIFY_ITER_RESIDUAL) {
        const int nbt = base(2) <= room ? 2 : 1;
        return Kn6Layout{nbt, 0, base(nbt)};
    }
    const size_t kids = (((size_t)Mmax * 24) + 127) & ~(size_t)127;
    const size_t pre = MISC_BYTES + tree + kids;
    const long long left = (long long)room - (long long)pre;
    long long cap = left > 0 ? left / 8 : 0;
    if (cap > chunk) cap = chunk;
    if (cap < NT) cap = 0;  // too few to help: recompute
    const size_t body = 2 * buf > (size_t)cap * 8 ? 2 * buf : (size_t)cap * 8;
    return Kn6Layout{1, (int)cap, pre + body};
}

}  // namespace

cudaError_t dt_kn6_set_probe(long long budget) {
    return cudaMemcpyToSymbol(g_kn6_probe, &budget, sizeof(budget));
}

size_t dt_kn6_smem_bytes(int chunk, int esize, int Mmax, int rule) {
    return kn6_layout(chunk, esize, Mmax, rule).total;
}

int dt_kn6_pq_cache(int chunk, int esize, int Mmax, int rule) {
    return kn6_layout(chunk, esize, Mmax, rule).cap;
}

// Sets the kernel's shared-memory and cluster-size attributes for a launch.
template <typename T, int RULE, bool CORR>
cudaError_t kn6_prepare(int S, size_t smem) {
    cudaError_t e =
        cudaFuncSetAttribute(kn6_kernel<T, RULE, CORR>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && S > 8)
        e = cudaFuncSetAttribute(kn6_kernel<T, RULE, CORR>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <typename T, int RULE, bool CORR>
int kn6_max_clusters(int S, size_t smem) {
    if (kn6_prepare<T, RULE, CORR>(S, smem) != cudaSuccess) return 0;
    return dt_max_active_clusters(kn6_kernel<T, RULE, CORR>, S, NT, smem);
}

template <typename T>
int kn6_max_clusters_rule(int rule, int S, size_t smem) {
    switch (rule) {
        case DT_VERIFY_GREEDY: return kn6_max_clusters<T, DT_VERIFY_GREEDY, false>(S, smem);
        case DT_VERIFY_RATIO: return kn6_max_clusters<T, DT_VERIFY_RATIO, false>(S, smem);
        case DT_VERIFY_ITER_RESIDUAL: return kn6_max_clusters<T, DT_VERIFY_ITER_RESIDUAL, false>(S, smem);
        case DT_VERIFY_TARGET_MATCH: return kn6_max_clusters<T, DT_VERIFY_TARGET_MATCH, false>(S, smem);
        default: return kn6_max_clusters<T, DT_VERIFY_RATIO, true>(S, smem);  // DT_KN6_RATIO_MARKOV
    }
}

template <typename T, int RULE, bool CORR>
cudaError_t kn6_launch_t(const DtLaunch& lc, size_t smem, int S, const Kn6Corr& corr, int L, int V, int Mmax,
                         int chunk, int nbt, int pq_cap, const int32_t* tok, const int32_t* parent,
                         const int32_t* depth, const int32_t* rank, const int32_t* n_nodes, const float* draft_lse,
                         const void* target, const float* target_lse, const void* draft, const float* uniforms,
                         int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok, float* visited_lse,
                         int32_t* status) {
    cudaError_t e = kn6_prepare<T, RULE, CORR>(S, smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&lc.cfg, kn6_kernel<T, RULE, CORR>, corr, L, V, Mmax, chunk, nbt, pq_cap, tok, parent,
                              depth, rank, n_nodes, draft_lse, (const T*)target, target_lse, (const T*)draft,
                              uniforms, acc_nodes, acc_len, next_tok, visited_lse, status);
}

template <typename T>
cudaError_t kn6_launch_rule(int rule, const DtLaunch& lc, size_t smem, int S, const Kn6Corr& corr, int L, int V,
                            int Mmax, int chunk, int nbt, int pq_cap, const int32_t* tok, const int32_t* parent,
                            const int32_t* depth, const int32_t* rank, const int32_t* n_nodes,
                            const float* draft_lse, const void* target, const float* target_lse, const void* draft,
                            const float* uniforms, int32_t* acc_nodes, int32_t* acc_len, int32_t* next_tok,
                            float* visited_lse, int32_t* status) {
#define DT_KN6_ARGS lc, smem, S, corr, L, V, Mmax, chunk, nbt, pq_cap, tok, parent, depth, rank, n_nodes, draft_lse, \
                    target, target_lse, draft, uniforms, acc_nodes, acc_len, next_tok, visited_lse, status
    switch (rule) {
        case DT_VERIFY_GREEDY: return kn6_launch_t<T, DT_VERIFY_GREEDY, false>(DT_KN6_ARGS);
        case DT_VERIFY_RATIO: return kn6_launch_t<T, DT_VERIFY_RATIO, false>(DT_KN6_ARGS);
        case DT_VERIFY_ITER_RESIDUAL: return kn6_launch_t<T, DT_VERIFY_ITER_RESIDUAL, false>(DT_KN6_ARGS);
        case DT_VERIFY_TARGET_MATCH: return kn6_launch_t<T, DT_VERIFY_TARGET_MATCH, false>(DT_KN6_ARGS);
        default: return kn6_launch_t<T, DT_VERIFY_RATIO, true>(DT_KN6_ARGS);
    }
#undef DT_KN6_ARGS
}

int dt_kn6_max_clusters(int dtype, int S, int chunk, int Mmax, int rule) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const size_t smem = dt_kn6_smem_bytes(chunk, esize, Mmax, rule);
    return dtype == DT_BF16 ? kn6_max_clusters_rule<uint16_t>(rule, S, smem)
                            : kn6_max_clusters_rule<float>(rule, S, smem);
}

cudaError_t dt_kn6_launch(int batch, int L, int V, int dtype, int Mmax, int S, int chunk, int rule,
                          const int32_t* tok, const int32_t* parent, const int32_t* depth, const int32_t* rank,
                          const int32_t* n_nodes, const float* draft_lse, const void* target,
                          const float* target_lse, const void* draft, const float* uniforms, int32_t* acc_nodes,
                          int32_t* acc_len, int32_t* next_tok, float* visited_lse, int32_t* status,
                          const DtKn6Proposal* prop, cudaStream_t st) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const Kn6Layout lay = kn6_layout(chunk, esize, Mmax, rule);
    const size_t smem = lay.total;
    const int nbt = lay.nbt, pq_cap = lay.cap;
    DtLaunch lc(dim3(S, batch, 1), dim3(NT, 1, 1), smem, st, S);
    Kn6Corr corr{nullptr, nullptr, 0, nullptr, 0, nullptr};
    if (rule == DT_KN6_RATIO_MARKOV) {
        if (!prop || !prop->U || !prop->Vt || prop->R < 4 || prop->R > 64 || (prop->R & 3) || !prop->z)
            return cudaErrorInvalidValue;
        corr = Kn6Corr{prop->U, prop->Vt, prop->R, prop->z, prop->K, prop->root_tok};
    }
    if (dtype == DT_BF16)
        return kn6_launch_rule<uint16_t>(rule, lc, smem, S, corr, L, V, Mmax, chunk, nbt, pq_cap, tok, parent, depth,
                                         rank, n_nodes, draft_lse, target, target_lse, draft, uniforms, acc_nodes,
                                         acc_len, next_tok, visited_lse, status);
    return kn6_launch_rule<float>(rule, lc, smem, S, corr, L, V, Mmax, chunk, nbt, pq_cap, tok, parent, depth, rank,
                                  n_nodes, draft_lse, target, target_lse, draft, uniforms, acc_nodes, acc_len,
                                  next_tok, visited_lse, status);
}
