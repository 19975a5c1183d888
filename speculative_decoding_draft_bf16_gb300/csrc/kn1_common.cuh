// kn1_common.cuh -- selection steps shared by the two stage-1 kernels.
#pragma once

#include "dt_device.cuh"

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
