// kn1_common.cuh -- selection steps shared by the two stage-1 kernels.
#pragma once

#include "dt_device.cuh"

// Folds a vector (values x, maximum vm) into a running (max M, sum S of
// exp(x - M)).  For |M| < 64 each term is exp2(x * log2e - c) with c = M *
// log2e rounded, one fused multiply-add: c's rounding error (<= 2^-18) is a
// factor common to all terms, shifting the log-normaliser by < 3e-6.  Larger
// maxima round x - M first, so that an element equal to M adds exactly 1 at
// any magnitude.
template <int EPV>
DT_DI void dt_online_add(const float (&x)[EPV], float vm, float& M, float& S) {
    const float NEG_INF = -__int_as_float(0x7F800000);
    const float log2e = 1.44269504088896340736f;
    if (vm > M) {
        S = (M == NEG_INF) ? 0.f : __fmul_rn(S, dt_ex2_approx(__fmul_rn(__fsub_rn(M, vm), log2e)));
        M = vm;
    }
    if (fabsf(M) < 64.f) {
        // two lanes per packed f32x2 instruction; with 8 or more elements two
        // independent accumulators shorten the dependent chain
        const float c = __fmul_rn(M, log2e);
        const unsigned long long l2 = dt_f2_pack(log2e, log2e), c2 = dt_f2_pack(-c, -c);
        unsigned long long acc[2] = {dt_f2_pack(0.f, 0.f), dt_f2_pack(0.f, 0.f)};
#pragma unroll
        for (int s = 0; s < EPV; s += 2) {
            float d0, d1;
            dt_f2_unpack(dt_f2_fma(dt_f2_pack(x[s], x[s + 1]), l2, c2), d0, d1);
            unsigned long long& a = acc[EPV >= 8 ? (s >> 1) & 1 : 0];
            a = dt_f2_add(a, dt_f2_pack(dt_ex2_approx(d0), dt_ex2_approx(d1)));
        }
        float a0, a1;
        dt_f2_unpack(EPV >= 8 ? dt_f2_add(acc[0], acc[1]) : acc[0], a0, a1);
        S = __fadd_rn(S, __fadd_rn(a0, a1));
        return;
    }
    if (M == NEG_INF) return;  // every element so far is -inf
    float e[EPV];
#pragma unroll
    for (int s = 0; s < EPV; ++s) e[s] = dt_ex2_approx(__fmul_rn(__fsub_rn(x[s], M), log2e));
#pragma unroll
    for (int w = EPV / 2; w > 0; w >>= 1)
#pragma unroll
        for (int s = 0; s < w; ++s) e[s] = __fadd_rn(e[s], e[s + w]);
    S = __fadd_rn(S, e[0]);
}

// Merges a running (max M2, sum S2 of exp(x - M2)) into (M, S).
DT_DI void dt_online_merge(float& M, float& S, float M2, float S2) {
    const float NEG_INF = -__int_as_float(0x7F800000);
    const float log2e = 1.44269504088896340736f;
    if (M2 == NEG_INF) return;
    if (M == NEG_INF) {
        M = M2;
        S = S2;
        return;
    }
    if (M2 > M) {
        S = __fadd_rn(__fmul_rn(S, dt_ex2_approx(__fmul_rn(__fsub_rn(M, M2), log2e))), S2);
        M = M2;
    } else {
        S = __fadd_rn(S, __fmul_rn(S2, dt_ex2_approx(__fmul_rn(__fsub_rn(M2, M), log2e))));
    }
}

// Shared-memory scratch of dt_find_bin.
struct DtBinSearch {
    int wsum[8];
    int digit;  // bin holding the need-th largest key, -1 if the bins hold fewer keys
    int need;   // keys still needed inside that bin
};

// Block-wide (NT >= 256 threads): in the 256-bin histogram g, find the bin
// holding the need-th largest key.  When TOP_IS_HIGH a higher bin index is a
// larger key, else bin 0 is the largest.  Results in bs->digit, bs->need.
// Contains two __syncthreads.
template <bool TOP_IS_HIGH>
DT_DI void dt_find_bin(const uint32_t* g, int need, DtBinSearch* bs) {
    const int t = threadIdx.x;
    int v = 0;
    if (t < 256) v = (int)g[TOP_IS_HIGH ? 255 - t : t];
    const int inc = dt_warp_incl_scan(v);
    if (t < 256 && (t & 31) == 31) bs->wsum[t >> 5] = inc;
    if (t == 0) {
        bs->digit = -1;
        bs->need = need;
    }
    __syncthreads();
    if (t < 256) {
        int before = 0;
        for (int i = 0; i < (t >> 5); ++i) before += bs->wsum[i];
        const int cum = before + inc;
        if (cum >= need && cum - v < need) {
            bs->digit = TOP_IS_HIGH ? 255 - t : t;
            bs->need = need - (cum - v);
        }
    }
    __syncthreads();
}

// Candidate entries are (order key << 32) | (0xFFFFFFFF - token id): distinct,
// and larger means ranked first (logit descending, token id ascending).
template <typename T>
DT_DI void dt_write_cand(unsigned long long key, int rank, int Kc, float lse, int row, int32_t* cand_id,
                         float* cand_lp) {
    cand_id[(size_t)row * Kc + rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
    cand_lp[(size_t)row * Kc + rank] = __fsub_rn(DtElem<T>::key_val((uint32_t)(key >> 32)), lse);
}

// Rank each of the `mine` entries `own` among the `total` entries `all` of the
// row and write those of rank < Kc.  One warp per entry.
template <typename T, int NT>
DT_DI void dt_rank_and_write(const unsigned long long* own, int mine, const unsigned long long* all, int total,
                             int Kc, float lse, int row, int32_t* cand_id, float* cand_lp) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = wid; i < mine; i += NT / 32) {
        const unsigned long long key = own[i];
        int rank = 0;
        for (int q = lane; q < total; q += 32) rank += (all[q] > key);
        rank = dt_warp_sum_i(rank);
        if (lane == 0 && rank < Kc) dt_write_cand<T>(key, rank, Kc, lse, row, cand_id, cand_lp);
    }
}

// The same with sixteen threads per entry (each counts a stride-16 slice of
// `all`, then a 4-step reduction within the half-warp): more entries in flight
// than one warp per entry when the lists are short.
template <typename T, int NT>
DT_DI void dt_rank16_and_write(const unsigned long long* own, int mine, const unsigned long long* all, int total,
                               int Kc, float lse, int row, int32_t* cand_id, float* cand_lp) {
    const int sub = threadIdx.x & 15, grp = threadIdx.x >> 4;
    const int rounds = (mine + NT / 16 - 1) / (NT / 16);
    for (int rd = 0; rd < rounds; ++rd) {  // uniform trip count: every lane reaches the shuffles
        const int i = grp + rd * (NT / 16);
        const bool live = i < mine;
        const unsigned long long key = live ? own[i] : ~0ull;
        int rank = 0;
        if (live)
            for (int q = sub; q < total; q += 16) rank += (all[q] > key);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (live && sub == 0 && rank < Kc) dt_write_cand<T>(key, rank, Kc, lse, row, cand_id, cand_lp);
    }
}

// Sort the row's `total` entries `all` (room for the next power of two),
// larger first, and write ranks [c*per, (c+1)*per) of the top Kc, per =
// ceil(Kc / S) -- with S CTAs on a row each writes its share.  For many
// entries, where ranking each against all others would cost more.
template <typename T, int NT>
DT_DI void dt_sort_and_write(unsigned long long* all, int total, int Kc, int c, int S, float lse, int row,
                             int32_t* cand_id, float* cand_lp) {
    const int n = dt_pow2_ceil(total);
    for (int i = total + threadIdx.x; i < n; i += NT) all[i] = 0ull;  // real entries are nonzero
    __syncthreads();
    dt_bitonic_u64<NT>(all, n, true);
    const int per = (Kc + S - 1) / S;
    const int r1 = min(min(Kc, total), (c + 1) * per);
    for (int r = c * per + threadIdx.x; r < r1; r += NT) dt_write_cand<T>(all[r], r, Kc, lse, row, cand_id, cand_lp);
}

// Entries of a row above which dt_sort_and_write replaces dt_rank_and_write.
constexpr int DT_SORT_MIN = 384;

// Shared-memory scratch of dt_bucket_rank_and_write.
struct DtRankScratch {
    uint32_t hist[256];
    uint32_t start[257];
    uint32_t fill[256];
    int wsum[8];
    int outside;
};

// Rank by key buckets.  The row's entries all[0, total) (distinct, larger
// first) go into 256 buckets by the top 16 bits of their order key, bucket b
// holding top16 - b (top16: those of the row maximum); an entry's rank is the
// number of entries in earlier buckets plus those of its own bucket with a
// larger key.  Entries [own_lo, own_hi) of rank < Kc are written.  The work
// is O(total + sum of squared bucket sizes).  Returns false, having written
// nothing, when an entry falls outside the 256 buckets (the caller sorts
// instead).  `bucket` has room for `total` entries.  Block-uniform; contains
// __syncthreads.
template <typename T, int NT>
DT_DI bool dt_bucket_rank_and_write(const unsigned long long* all, int total, int own_lo, int own_hi, uint32_t top16,
                                    int Kc, float lse, int row, int32_t* cand_id, float* cand_lp,
                                    DtRankScratch* rs, unsigned long long* bucket) {
    constexpr int SH = 32 + DtElem<T>::KB - 16;  // entry bits above which the key's top 16 bits sit
    const int t = threadIdx.x, lane = t & 31;
    if (t < 256) {
        rs->hist[t] = 0;
        rs->fill[t] = 0;
    }
    if (t == 0) rs->outside = 0;
    __syncthreads();
    for (int i = t; i < total; i += NT) {
        const uint32_t b = top16 - (uint32_t)(all[i] >> SH);
        if (b < 256u) atomicAdd(&rs->hist[b], 1u);
        else rs->outside = 1;
    }
    __syncthreads();
    if (rs->outside) return false;
    // exclusive scan of the bucket sizes
    int v = 0, inc = 0;
    if (t < 256) {
        v = (int)rs->hist[t];
        inc = dt_warp_incl_scan(v);
        if (lane == 31) rs->wsum[t >> 5] = inc;
    }
    __syncthreads();
    if (t < 256) {
        int before = 0;
        for (int w = 0; w < (t >> 5); ++w) before += rs->wsum[w];
        rs->start[t] = (uint32_t)(before + inc - v);
        if (t == 255) rs->start[256] = (uint32_t)(before + inc);
    }
    __syncthreads();
    for (int i = t; i < total; i += NT) {
        const unsigned long long key = all[i];
        const uint32_t b = top16 - (uint32_t)(key >> SH);
        bucket[rs->start[b] + atomicAdd(&rs->fill[b], 1u)] = key;
    }
    __syncthreads();
    for (int i = own_lo + t; i < own_hi; i += NT) {
        const unsigned long long key = all[i];
        const uint32_t b = top16 - (uint32_t)(key >> SH);
        const int q0 = (int)rs->start[b], q1 = (int)rs->start[b + 1];
        int r = q0;
        for (int q = q0; q < q1; ++q) r += (bucket[q] > key);
        if (r < Kc) dt_write_cand<T>(key, r, Kc, lse, row, cand_id, cand_lp);
    }
    return true;
}
