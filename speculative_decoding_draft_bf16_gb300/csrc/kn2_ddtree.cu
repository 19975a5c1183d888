// kn2_ddtree.cu -- DDTree Top-B selection over the S_K prefix set.
//
// [DDTree] Prop 2 (a prefix is at least as likely as its extensions), Lemma
// (S_K) and Algorithm 1 (best-first heap over rank descriptors); [DARTree]
// "Tree verification and DDTree".  The heap pops the B best prefixes of S_K
// under the node order (score descending, then rank descriptor ascending with
// a prefix first); score = lp_1[rho_1] + ... + lp_d[rho_d] in fp32, added from
// the root's 0.  Because a child never outscores its parent and a later
// sibling never outscores an earlier one, that order places every prefix
// after its predecessor, and the popped set is exactly the B smallest prefixes
// in the order.
//
// GPU formulation (no heap): one CTA per request keeps C = the B best prefixes
// of depth <= d, sorted.  C for depth d is the best B of C(d-1) plus the
// children of C(d-1)'s depth-(d-1) nodes, since every depth-d member of the
// answer has its parent there.  Per depth: list those parents in
// lexicographic order, count per parent the children that can still enter
// (binary search against the current B-th score; each parent's children are
// sorted), materialise them as 64-bit keys (score, lexicographic position),
// sort, and merge with C (merge path: one binary search per element).  Ties
// across depths are resolved by walking the candidate's ancestors.  Stops at
// the first depth that adds nothing.  Work per depth is O((|C| + m) log) plus
// the sorts (up to 512 keys: warp-register sorts of 32-key segments ranked
// against each other by binary search, two block barriers); everything lives
// in shared memory.  A per-request budget (budget[b], clamped to [1, B], e.g.
// from SABA) replaces B for that request; the buffers keep B's stride.
#include "dt_device.cuh"
#include "dt_mask.cuh"
#include "dt_launch.h"

namespace {

// Threads per request (measured on a GB300, single request, B = K = 256:
// select 8.25 / 7.28 / 7.60 us with 128 / 256 / 512 threads).
#ifndef DT_KN2_NT
#define DT_KN2_NT 256
#endif
constexpr int NT = DT_KN2_NT;
constexpr int CAP = 2048;  // candidates materialised per merge
constexpr int SMALL_M = 256;  // merges of at most this many candidates rank them without a sort
static_assert(SMALL_M * 8 + SMALL_M * 4 * 2 <= CAP * 8, "the small-merge arrays must fit after its keys");

struct Kn2Smem {
    float* lp;       // [K]
    float* cs;       // [2][B] scores (buffer `cur` at offset cur*B)
    int* cpar;       // [2][B] parent C index (-1 = root)
    int* crank;      // [2][B]
    int* cdep;       // [2][B]
    uint32_t* clex;  // [2][B] (lexrank of parent << 16) | rank
    int* pidx;       // [B] parents in lexicographic order (C index or -1)
    int* pn;         // [B + 1]
    int* newpos;     // [B]
    unsigned long long* cand;  // [CAP]
};

// All positions' lp rows are staged up front when they fit in this budget.
constexpr int LP_ALL_BYTES = 64 * 1024;

DT_DI Kn2Smem carve(unsigned char* s, int L, int K, int B) {
    Kn2Smem m;
    m.cand = (unsigned long long*)s;
    s += (size_t)CAP * 8;
    m.lp = (float*)s;
    const int rows = ((size_t)L * K * 4 <= LP_ALL_BYTES) ? L : 1;
    s += (size_t)((rows * K + 3) & ~3) * 4;
    m.cs = (float*)s; s += (size_t)2 * B * 4;
    m.cpar = (int*)s; s += (size_t)2 * B * 4;
    m.crank = (int*)s; s += (size_t)2 * B * 4;
    m.cdep = (int*)s; s += (size_t)2 * B * 4;
    m.clex = (uint32_t*)s; s += (size_t)2 * B * 4;
    m.pidx = (int*)s; s += (size_t)B * 4;
    m.newpos = (int*)s; s += (size_t)B * 4;
    m.pn = (int*)s;
    return m;
}

// Does C node i precede the depth-d candidate with key y?
DT_DI bool c_before_cand(int i, unsigned long long y, int d, const float* cs, const int* cdep, const int* cpar,
                         const uint32_t* clex, const int* pidx) {
    // score keys, not floats: a strict total order even for NaN scores
    const uint32_t ky = (uint32_t)(y >> 32), ki = dt_fkey(cs[i]);
    if (ki != ky) return ki > ky;
    const uint32_t ly = 0xFFFFFFFFu - (uint32_t)y;
    const int e = cdep[i];
    if (e == d) return clex[i] < ly;
    int a = pidx[ly >> 16];
    while (cdep[a] > e) a = cpar[a];
    if (a == i) return true;  // C node i is an ancestor of the candidate
    return clex[i] < clex[a];
}

__global__ void __launch_bounds__(NT, 1) kn2_kernel(const float* __restrict__ cand_lp,
                                                 const int32_t* __restrict__ cand_id,
                                                 const float* __restrict__ lse, int L, int K, int Bcap,
                                                 const int32_t* __restrict__ budget, int Mmax,
                                                 int32_t* __restrict__ o_tok, int32_t* __restrict__ o_par,
                                                 int32_t* __restrict__ o_dep, int32_t* __restrict__ o_rank,
                                                 float* __restrict__ o_score, int32_t* __restrict__ o_n,
                                                 int32_t* __restrict__ status, uint32_t* __restrict__ o_mask,
                                                 int32_t* __restrict__ o_pos, int pos_offset) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int red[NT / 32];
    __shared__ int sh_nP, sh_lrhi, sh_any;
    __shared__ float chain[DT_MAX_L + 1];  // score of the rank-0 chain to each depth
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    Kn2Smem S = carve(smem, L, K, Bcap);
    dt_pdl_trigger();
    dt_pdl_wait();
    // this request's budget (buffers are sized for Bcap)
    const int B = budget ? min(Bcap, max(1, budget[b])) : Bcap;
    const float* lpb = cand_lp + (size_t)b * L * K;
    const bool lp_all = (size_t)L * K * 4 <= LP_ALL_BYTES;
    if (lp_all)
        for (int i = tid; i < L * K; i += NT) S.lp[i] = lpb[i];
    if (tid == 0) {
        // every depth-d prefix scores at most the rank-0 chain (lp is sorted
        // within a position and fp32 addition is monotone)
        float u = 0.f;
        chain[0] = 0.f;
        for (int d = 1; d <= L; ++d) {
            u = __fadd_rn(u, lpb[(size_t)(d - 1) * K]);
            chain[d] = u;
        }
    }

    // depth 1: the root's children are the first min(K, B) ranks, already in order
    int nC = min(K, B);
    int cur = 0;
    for (int i = tid; i < nC; i += NT) {
        S.cs[i] = lpb[i];
        S.cpar[i] = -1;
        S.crank[i] = i;
        S.cdep[i] = 1;
        S.clex[i] = (uint32_t)i;
    }
    __syncthreads();

    for (int d = 2; d <= L; ++d) {
        const bool full0 = (nC == B);
        const float tau0 = full0 ? (S.cs + cur * Bcap)[B - 1] : 0.f;
        // nothing at this depth or below can reach the current B-th score
        if (full0 && chain[d] < tau0) break;
        const float* lpd = S.lp;
        if (lp_all) {
            lpd = S.lp + (size_t)(d - 1) * K;
        } else {
            __syncthreads();
            for (int r = tid; r < K; r += NT) S.lp[r] = lpb[(size_t)(d - 1) * K + r];
            __syncthreads();
        }
        // ---- parents: depth-(d-1) members of C whose best child can still
        // enter, in lexicographic order ----------------------------------------
        {
            const float lp0 = lpd[0];
            int cnt_local = 0;
            for (int i = tid; i < nC; i += NT)
                cnt_local += ((S.cdep + cur * Bcap)[i] == d - 1) &&
                             (!full0 || __fadd_rn((S.cs + cur * Bcap)[i], lp0) >= tau0);
            // compact with a scan over a per-thread strided layout
            int tot;
            int ex = dt_block_excl_scan<NT>(cnt_local, red, &tot);
            int w = ex;
            for (int i = tid; i < nC; i += NT)
                if ((S.cdep + cur * Bcap)[i] == d - 1 && (!full0 || __fadd_rn((S.cs + cur * Bcap)[i], lp0) >= tau0))
                    S.cand[w++] = ((unsigned long long)(S.clex + cur * Bcap)[i] << 32) | (unsigned)i;
            if (tid == 0) { sh_nP = tot; sh_any = 0; }
            __syncthreads();
            // already in lexicographic order? then no sort.  The depth-1 nodes
            // always are when each thread compacted at most one of them: their
            // scores fall with their rank, so C holds them in rank order.
            if (d > 2 || nC > NT) {
                for (int i = tid; i + 1 < tot; i += NT)
                    if (S.cand[i] > S.cand[i + 1]) sh_any = 1;
                __syncthreads();
            }
            if (sh_any) {
                if (tot <= 32) {
                    dt_warp_sort_u64(S.cand, tot, false);
                } else if (tot <= 512) {
                    dt_block_sort_u64<NT>(S.cand, tot, false, S.cand + 512);
                } else {
                    const int P2 = dt_pow2_ceil(tot);
                    for (int i = tot + tid; i < P2; i += NT) S.cand[i] = ~0ull;
                    __syncthreads();
                    dt_bitonic_u64<NT>(S.cand, P2, false);
                }
            }
            for (int j = tid; j < tot; j += NT) S.pidx[j] = (int)(S.cand[j] & 0xFFFFFFFFull);
            __syncthreads();
        }
        const int nP = sh_nP;
        if (nP == 0) break;

        int lr_lo = 0;
        while (lr_lo < nP) {
            const bool full = (nC == B);
            const float tau = full ? (S.cs + cur * Bcap)[B - 1] : 0.f;
            // children of each remaining parent that can still enter
            for (int j = tid; j < nP; j += NT) {
                int cnt = 0;
                const int p = S.pidx[j];
                if (j >= lr_lo && p >= 0) {
                    if (!full) {
                        cnt = K;
                    } else {
                        const float sp = (S.cs + cur * Bcap)[p];
                        int lo = 0, hi = K;
                        while (lo < hi) {
                            int mid = (lo + hi) >> 1;
                            if (__fadd_rn(sp, lpd[mid]) >= tau) lo = mid + 1;
                            else hi = mid;
                        }
                        cnt = lo;
                    }
                    cnt = min(cnt, B);
                }
                S.pn[j] = cnt;
            }
            __syncthreads();
            dt_block_scan_array<NT>(S.pn, S.pn, nP, red);
            int lr_hi = nP;  // the rest of the parents, when their children fit CAP
            if (S.pn[nP] - S.pn[lr_lo] > CAP) {  // block-uniform
                if (tid == 0) sh_lrhi = lr_lo + 1;
                __syncthreads();
                for (int j = lr_lo + 1 + tid; j <= nP; j += NT)
                    if (S.pn[j] - S.pn[lr_lo] <= CAP) atomicMax(&sh_lrhi, j);
                __syncthreads();
                lr_hi = sh_lrhi;
            }
            const int base = S.pn[lr_lo];
            const int m = S.pn[lr_hi] - base;
            if (m > 0) {
                // materialise candidates (key: score, then lexicographic position)
                for (int idx = tid; idx < m; idx += NT) {
                    const int g = base + idx;
                    int lo = lr_lo, hi = lr_hi;  // find j with pn[j] <= g < pn[j+1]
                    while (hi - lo > 1) {
                        int mid = (lo + hi) >> 1;
                        if (S.pn[mid] <= g) lo = mid;
                        else hi = mid;
                    }
                    const int j = lo;
                    const int r = g - S.pn[j];
                    const float s = __fadd_rn((S.cs + cur * Bcap)[S.pidx[j]], lpd[r]);
                    const uint32_t lex = ((uint32_t)j << 16) | (uint32_t)r;
                    S.cand[idx] = ((unsigned long long)dt_fkey(s) << 32) | (unsigned long long)(0xFFFFFFFFu - lex);
                }
                __syncthreads();
                const int nx = cur ^ 1;
                const float* ccs = S.cs + cur * Bcap;
                const int* ccdep = S.cdep + cur * Bcap;
                const int* ccpar = S.cpar + cur * Bcap;
                const uint32_t* cclex = S.clex + cur * Bcap;
                // C members before candidate y (C is sorted, the predicate monotone)
                auto c_before = [&](unsigned long long y) {
                    int lo = 0, hi = nC;
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (c_before_cand(mid, y, d, ccs, ccdep, ccpar, cclex, S.pidx)) lo = mid + 1;
                        else hi = mid;
                    }
                    return lo;
                };
                // a candidate's new position: its rank among the candidates plus
                // the C members before it
                int* cpos = (int*)(S.cand + SMALL_M);  // [SMALL_M] C members before candidate q
                int* cfin = cpos + SMALL_M;           // [SMALL_M] its position in the merged order
                if (m <= SMALL_M) {
                    // no sort: rank each candidate against all (keys are
                    // distinct), and move C member i by the candidates placed
                    // before it
                    for (int q = tid; q < m; q += NT) {
                        const unsigned long long y = S.cand[q];
                        int r = 0;
                        for (int q2 = 0; q2 < m; ++q2) r += (S.cand[q2] > y);
                        const int lo = c_before(y);
                        cpos[q] = lo;
                        cfin[q] = r + lo;
                    }
                    __syncthreads();
                    for (int i = tid; i < nC; i += NT) {
                        int before = 0;
                        for (int q = 0; q < m; ++q) before += (cpos[q] <= i);
                        const int nr = i + before;
                        S.newpos[i] = nr < B ? nr : -1;
                    }
                } else {
                    if (m <= 512) {
                        dt_block_sort_u64<NT>(S.cand, m, true, S.cand + 512);
                    } else {
                        const int P2 = dt_pow2_ceil(m);
                        for (int i = m + tid; i < P2; i += NT) S.cand[i] = 0ull;
                        __syncthreads();
                        dt_bitonic_u64<NT>(S.cand, P2, true);
                    }
                    const int mm = min(m, B);
                    // merge path: new position of every C member ...
                    for (int i = tid; i < nC; i += NT) {
                        int lo = 0, hi = mm;
                        while (lo < hi) {
                            int mid = (lo + hi) >> 1;
                            if (c_before_cand(i, S.cand[mid], d, ccs, ccdep, ccpar, cclex, S.pidx))
                                hi = mid;
                            else
                                lo = mid + 1;
                        }
                        const int nr = i + lo;
                        S.newpos[i] = nr < B ? nr : -1;
                    }
                }
                __syncthreads();
                for (int i = tid; i < nC; i += NT) {
                    const int np = S.newpos[i];
                    if (np >= 0) {
                        const int pp = ccpar[i];
                        (S.cs + nx * Bcap)[np] = ccs[i];
                        (S.cpar + nx * Bcap)[np] = pp < 0 ? -1 : S.newpos[pp];
                        (S.crank + nx * Bcap)[np] = (S.crank + cur * Bcap)[i];
                        (S.cdep + nx * Bcap)[np] = ccdep[i];
                        (S.clex + nx * Bcap)[np] = cclex[i];
                    }
                }
                // ... and of every candidate that still enters
                const int mq = m <= SMALL_M ? m : min(m, B);
                for (int q = tid; q < mq; q += NT) {
                    const unsigned long long y = S.cand[q];
                    const int nr = m <= SMALL_M ? cfin[q] : q + c_before(y);
                    if (nr < B) {
                        const uint32_t lex = 0xFFFFFFFFu - (uint32_t)y;
                        const int j = (int)(lex >> 16);
                        (S.cs + nx * Bcap)[nr] = dt_fkey_val((uint32_t)(y >> 32));
                        (S.cpar + nx * Bcap)[nr] = S.newpos[S.pidx[j]];
                        (S.crank + nx * Bcap)[nr] = (int)(lex & 0xFFFFu);
                        (S.cdep + nx * Bcap)[nr] = d;
                        (S.clex + nx * Bcap)[nr] = lex;
                    }
                }
                __syncthreads();
                for (int j = tid; j < nP; j += NT) {
                    const int p = S.pidx[j];
                    if (p >= 0) S.pidx[j] = S.newpos[p];
                }
                nC = min(B, nC + m);
                cur = nx;
                __syncthreads();
            }
            lr_lo = lr_hi;
        }
        // stop once a depth adds nothing
        if (tid == 0) sh_any = 0;
        __syncthreads();
        for (int i = tid; i < nC; i += NT)
            if ((S.cdep + cur * Bcap)[i] == d) sh_any = 1;
        __syncthreads();
        if (!sh_any) break;
    }

    // ---- output: root, then C in order -----------------------------------
    const size_t ob = (size_t)b * Mmax;
    for (int i = tid; i < nC; i += NT) {
        const int dd = (S.cdep + cur * Bcap)[i];
        const int rr = (S.crank + cur * Bcap)[i];
        o_tok[ob + i + 1] = cand_id[((size_t)b * L + dd - 1) * K + rr];
        o_par[ob + i + 1] = (S.cpar + cur * Bcap)[i] + 1;
        o_dep[ob + i + 1] = dd;
        o_rank[ob + i + 1] = rr;
        o_score[ob + i + 1] = (S.cs + cur * Bcap)[i];
        if (o_mask) o_pos[ob + i + 1] = dd + pos_offset;
    }
    if (tid == 0) {
        if (o_mask) o_pos[ob] = pos_offset;
        o_tok[ob] = -1;
        o_par[ob] = -1;
        o_dep[ob] = 0;
        o_rank[ob] = -1;
        o_score[ob] = 0.f;
        o_n[b] = nC + 1;
        int bits = 0;
        for (int l = 0; l < L; ++l) {
            const float v = lse[(size_t)b * L + l];
            if (v != v) bits |= DT_DEV_TIMEOUT;  // stage 1 flagged this row
        }
        status[b] = bits;
    }
    if (o_mask) {  // fused tree mask (positions above): parents from C in shared memory
        const int* cpar = S.cpar + cur * Bcap;
        dt_write_mask_rows<NT>(nC + 1, Mmax, [&](int a) { return a == 0 ? -1 : cpar[a - 1] + 1; },
                               o_mask + (size_t)b * Mmax * ((Mmax + 31) >> 5));
    }
}

}  // namespace

size_t dt_kn2_smem_bytes(int L, int K, int B) {
    const int rows = ((size_t)L * K * 4 <= LP_ALL_BYTES) ? L : 1;
    return (size_t)CAP * 8 + (size_t)((rows * K + 3) & ~3) * 4 + (size_t)B * 4 * 10 + (size_t)B * 8 +
           (size_t)(B + 1) * 4 + 16;
}

cudaError_t dt_kn2_launch(int batch, int L, int K, int B, const int32_t* budget, int Mmax, const float* cand_lp,
                          const int32_t* cand_id,
                          const float* lse, int32_t* tok, int32_t* parent, int32_t* depth, int32_t* rank,
                          float* score, int32_t* n_nodes, int32_t* status, uint32_t* mask, int32_t* pos,
                          int pos_offset, cudaStream_t st) {
    const size_t smem = dt_kn2_smem_bytes(L, K, B);
    cudaError_t e = cudaFuncSetAttribute(kn2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    DtLaunch lc(dim3(batch), dim3(NT), smem, st);
    return cudaLaunchKernelEx(&lc.cfg, kn2_kernel, cand_lp, cand_id, lse, L, K, B, budget, Mmax, tok, parent, depth, rank,
                              score, n_nodes, status, mask, pos, pos_offset);
}
