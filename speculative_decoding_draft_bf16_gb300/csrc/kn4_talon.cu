// kn4_talon.cu -- TALON budgeted, confidence-gated tree expansion.
//
// [TALON] key design 1: the root layer keeps the Top-k tokens of the first
// position regardless of confidence.  Key design 2: each later layer pools
// every child of the last layer, scores it by its path probability
// p(u) = p(v) * P(w) (log domain: s(u) = s(v) + lp(w), fp32), takes the anchor
// m_d = max p(u) over the pool and keeps p(u) >= mu * m_d (s >= m_d + log mu);
// if the layer passing the gate exceeds the remaining budget N - |T| it keeps
// only the best N - |T| (shared node order) and growth stops.  At most L
// layers.  For a block drafter P(w) is position d's marginal, so each
// position's Top-min(N, V) list suffices: a kept child of rank r needs its r
// better-ranked siblings kept as well.
//
// One CTA per request, everything in shared memory.  Layers are stored in
// lexicographic order (children materialised parent by parent in rank
// order), so a node's lexicographic key within its depth is
// (index of its parent within the parent layer << 16) | rank.  Per layer the
// passing children of each parent form a rank prefix found by binary search;
// on overflow the best N - |T| are chosen in groups of parents (running
// top list + group, bitonic sort), pruning later groups by the running cutoff.
// The finished tree is sorted once in the shared node order.
#include "dt_device.cuh"
#include "dt_mask.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT = 512;

struct Kn4Smem {
    float* lp;                 // [Kc]
    float* s;                  // [N]
    int* dep;
    int* par;
    int* rank;
    uint32_t* lex;
    int* pn;                   // [N + 1]
    int* ord;                  // [pow2(N)]
};

DT_DI Kn4Smem kn4_carve(unsigned char* p, int Kc, int N) {
    Kn4Smem m;
    m.lp = (float*)p; p += (size_t)((Kc + 3) & ~3) * 4;
    m.s = (float*)p; p += (size_t)N * 4;
    m.dep = (int*)p; p += (size_t)N * 4;
    m.par = (int*)p; p += (size_t)N * 4;
    m.rank = (int*)p; p += (size_t)N * 4;
    m.lex = (uint32_t*)p; p += (size_t)N * 4;
    m.pn = (int*)p; p += (size_t)(N + 1) * 4;
    m.ord = (int*)p;
    return m;
}

// Count of the first-ranked children w of a parent with score sp that satisfy
// sp + lp[w] >= thr (monotone in w).
DT_DI int count_pass(float sp, const float* lp, int Kc, float thr) {
    int lo = 0, hi = Kc;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__fadd_rn(sp, lp[mid]) >= thr) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Locate j with pn[j] <= g < pn[j+1] within [lo, hi).
DT_DI int find_parent(const int* pn, int lo, int hi, int g) {
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pn[mid] <= g) lo = mid;
        else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(NT, 1) kn4_kernel(int L, int Kc, int talon_k, float log_mu, int N, int Mmax,
                                                 const float* __restrict__ cand_lp,
                                                 const int32_t* __restrict__ cand_id, const float* __restrict__ lse,
                                                 int32_t* __restrict__ o_tok, int32_t* __restrict__ o_par,
                                                 int32_t* __restrict__ o_dep, int32_t* __restrict__ o_rank,
                                                 float* __restrict__ o_score, int32_t* __restrict__ o_n,
                                                 int32_t* __restrict__ status, uint32_t* __restrict__ o_mask,
                                                 int32_t* __restrict__ o_pos, int pos_offset) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int red[NT / 32];
    __shared__ float redf[NT / 32];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    Kn4Smem S = kn4_carve(smem, Kc, N);
    dt_pdl_trigger();
    dt_pdl_wait();
    const float* lpb = cand_lp + (size_t)b * L * Kc;

    // root layer: Top-k of position 1
    const int k1 = min(min(talon_k, Kc), N);
    for (int i = tid; i < k1; i += NT) {
        S.s[i] = lpb[i];
        S.dep[i] = 1;
        S.par[i] = -1;
        S.rank[i] = i;
        S.lex[i] = (uint32_t)i;
    }
    int nT = k1, lay_lo = 0, lay_hi = k1;
    for (int d = 2; d <= L && nT < N; ++d) {
        __syncthreads();
        for (int w = tid; w < Kc; w += NT) S.lp[w] = lpb[(size_t)(d - 1) * Kc + w];
        __syncthreads();
        const int nP = lay_hi - lay_lo;
        // anchor: best child score over the pool
        float mx = -__int_as_float(0x7F800000);
        for (int j = tid; j < nP; j += NT) mx = fmaxf(mx, __fadd_rn(S.s[lay_lo + j], S.lp[0]));
        mx = dt_warp_max(mx);
        if (lane == 0) redf[wid] = mx;
        __syncthreads();
        float m_d = redf[0];
        for (int w = 1; w < NT / 32; ++w) m_d = fmaxf(m_d, redf[w]);
        const float thr = __fadd_rn(m_d, log_mu);
        for (int j = tid; j < nP; j += NT) S.pn[j] = count_pass(S.s[lay_lo + j], S.lp, Kc, thr);
        __syncthreads();
        dt_block_scan_array<NT>(S.pn, S.pn, nP, red);
        const int m = S.pn[nP];
        const int room = N - nT;
        if (m <= room) {
            // the whole passing pool becomes the next layer, in lexicographic order
            for (int g = tid; g < m; g += NT) {
                const int j = find_parent(S.pn, 0, nP, g);
                const int w = g - S.pn[j];
                const int x = nT + g;
                S.s[x] = __fadd_rn(S.s[lay_lo + j], S.lp[w]);
                S.dep[x] = d;
                S.par[x] = lay_lo + j;
                S.rank[x] = w;
                S.lex[x] = ((uint32_t)j << 16) | (uint32_t)w;
            }
            lay_lo = nT;
            lay_hi = nT + m;
            nT += m;
            continue;
        }
        // overflow: keep the best `room` of the pool, then stop.  Every
        // parent's passing children are a rank prefix, so the number of pool
        // members scoring >= t is a sum of per-parent binary searches; a
        // binary search over the order keys of t in [thr, m_d] finds the
        // R-th best score t*.  The layer takes every member above t* and the
        // first ties at t* in lexicographic order (parent, then rank).
        const int R = room;
        auto count_all = [&](float t) {
            int c = 0;
            for (int j = tid; j < nP; j += NT) c += count_pass(S.s[lay_lo + j], S.lp, Kc, t);
            c = dt_warp_sum_i(c);
            if (lane == 0) red[wid] = c;
            __syncthreads();
            int tot = 0;
#pragma unroll
            for (int w = 0; w < NT / 32; ++w) tot += red[w];
            __syncthreads();
            return tot;
        };
        uint32_t klo = dt_fkey(thr), khi = dt_fkey(m_d) + 1u;  // count(klo) >= R > count(khi)
        while (khi - klo > 1u) {
            const uint32_t mid = klo + ((khi - klo) >> 1);
            if (count_all(dt_fkey_val(mid)) >= R) klo = mid;
            else khi = mid;
        }
        const float t_eq = dt_fkey_val(klo), t_gt = dt_fkey_val(klo + 1u);
        // per parent: a = children above t*, ties = children at t*
        for (int j = tid; j < nP; j += NT) {
            const int a_j = count_pass(S.s[lay_lo + j], S.lp, Kc, t_gt);
            S.pn[j] = count_pass(S.s[lay_lo + j], S.lp, Kc, t_eq) - a_j;
            S.ord[j] = a_j;
        }
        __syncthreads();
        dt_block_scan_array<NT>(S.pn, S.pn, nP, red);  // exclusive prefix of the ties
        {
            // ties still needed after every member above t*
            int c = 0;
            for (int j = tid; j < nP; j += NT) c += S.ord[j];
            c = dt_warp_sum_i(c);
            if (lane == 0) red[wid] = c;
            __syncthreads();
            int above = 0;
#pragma unroll
            for (int w = 0; w < NT / 32; ++w) above += red[w];
            const int need = R - above;
            __syncthreads();
            // parent j takes its a_j children above t* plus its share of ties
            for (int j = tid; j < nP; j += NT) {
                const int t0 = S.pn[j], tj = S.pn[j + 1] - t0;
                const int take_t = max(0, min(tj, need - t0));
                S.ord[j] += take_t;
            }
            __syncthreads();
        }
        dt_block_scan_array<NT>(S.ord, S.pn, nP, red);  // prefix of the per-parent takes
        const int nR = S.pn[nP];
        for (int g = tid; g < nR; g += NT) {
            const int j = find_parent(S.pn, 0, nP, g);
            const int w = g - S.pn[j];
            const int x = nT + g;
            S.s[x] = __fadd_rn(S.s[lay_lo + j], S.lp[w]);
            S.dep[x] = d;
            S.par[x] = lay_lo + j;
            S.rank[x] = w;
            S.lex[x] = ((uint32_t)j << 16) | (uint32_t)w;
        }
        nT += nR;
        break;
    }
    __syncthreads();

    // final order: root, then the shared node order
    const int Q2 = dt_pow2_ceil(nT);
    for (int q = tid; q < Q2; q += NT) S.ord[q] = q < nT ? q : -1;
    __syncthreads();
    dt_bitonic_nodes<NT>(S.ord, Q2, S.s, S.dep, S.par, S.lex);
    // output index of each node (reuse pn as the map)
    for (int q = tid; q < nT; q += NT) S.pn[S.ord[q]] = q + 1;
    __syncthreads();
    const size_t ob = (size_t)b * Mmax;
    for (int q = tid; q < nT; q += NT) {
        const int x = S.ord[q];
        const int dd = S.dep[x], rr = S.rank[x], p = S.par[x];
        o_tok[ob + q + 1] = cand_id[((size_t)b * L + dd - 1) * Kc + rr];
        o_par[ob + q + 1] = p < 0 ? 0 : S.pn[p];
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
        o_n[b] = nT + 1;
        int bits = 0;
        for (int l = 0; l < L; ++l) {
            const float x = lse[(size_t)b * L + l];
            if (x != x) bits |= DT_DEV_TIMEOUT;  // stage 1 flagged this row
        }
        status[b] = bits;
    }
    if (o_mask) {  // fused tree mask (positions above): parents through the output map in shared memory
        dt_write_mask_rows<NT>(nT + 1, Mmax,
                               [&](int a) {
                                   if (a == 0) return -1;
                                   const int p = S.par[S.ord[a - 1]];
                                   return p < 0 ? 0 : S.pn[p];
                               },
                               o_mask + (size_t)b * Mmax * ((Mmax + 31) >> 5));
    }
}

}  // namespace

size_t dt_kn4_smem_bytes(int Kc, int N) {
    int q2 = 1;
    while (q2 < N) q2 <<= 1;
    return (size_t)((Kc + 3) & ~3) * 4 + (size_t)N * 20 + (size_t)(N + 1) * 4 + (size_t)q2 * 4 + 16;
}

cudaError_t dt_kn4_launch(int batch, int L, int Kc, int talon_k, float log_mu, int N, int Mmax,
                          const float* cand_lp, const int32_t* cand_id, const float* lse, int32_t* tok,
                          int32_t* parent, int32_t* depth, int32_t* rank, float* score, int32_t* n_nodes,
                          int32_t* status, uint32_t* mask, int32_t* pos, int pos_offset, cudaStream_t st) {
    const size_t smem = dt_kn4_smem_bytes(Kc, N);
    cudaError_t e = cudaFuncSetAttribute(kn4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    DtLaunch lc(dim3(batch), dim3(NT), smem, st);
    return cudaLaunchKernelEx(&lc.cfg, kn4_kernel, L, Kc, talon_k, log_mu, N, Mmax, cand_lp, cand_id, lse, tok,
                              parent, depth, rank, score, n_nodes, status, mask, pos, pos_offset);
}
