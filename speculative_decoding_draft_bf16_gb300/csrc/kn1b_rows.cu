// kn1b_rows.cu -- stage 1 for batches of many rows: one CTA per row.
//
// [DARTree] Algorithm 1, its per-position Top-K candidate step; [DDTree] section 3.3
// (log-domain scores of each position's Top-K tokens).
//
// With enough rows (request b, position l) to fill the GPU, a whole row per
// CTA needs no cross-CTA exchange at all:
//   pass 1  streams the row from HBM: each thread copies its 16-byte
//           vectors (every NT-th) asynchronously into its own ring of RING
//           shared-memory slots (16 at one CTA per SM when every row has an SM
//           to itself, else 8 at two per SM), in pairs, RING - 2 copies in
//           flight, and keeps a running maximum and sum exp(x - max) (rescaled
//           whenever the maximum grows; the two vectors of each landed pair are
//           folded in together), and the maximum of its vectors m = u (mod
//           4) for u = 0..3 -- 4 x 512 = 2048 slot maxima of distinct
//           elements;
//   the CTA merges the (max, sum) pairs into the row's log-normaliser and
//   takes the Kc-th largest slot maximum (256-bin histogram of order keys
//   below the row maximum) as a lower bound for the row's Kc-th largest logit;
//   pass 2  re-reads only what can hold a candidate.  Short lists (Kc <=
//           KC_WORDS) re-read the slots whose maximum reaches the bound.
//           Longer ones, for which a slot is too coarse, have each thread
//           leave, in pass 1, a 16-bit word per vector (its maximum; one per
//           group of vectors on very long rows) in shared memory; pass 2 then
//           lists the vectors whose word reaches the bound in vector order
//           (one block scan over the word array) and re-reads only them --
//           about 1.4 Kc vectors instead of half the row at Kc = 1024 --
//           every thread a contiguous run of the list staged through shared
//           memory, so that the elements at or above the bound, placed with
//           a block scan, come out in token-id order;
//   the candidates are ranked exactly (logit descending, token id ascending):
//   up to 128 of them each against all (16 threads per candidate); more, on
//   bf16 words in id order, by a stable counting sort on the value (each of
//   256 buckets below the maximum is one bf16 value); else by key buckets or
//   a sort.  The top Kc are written.
// A row whose candidates overflow the buffer (many equal logits) takes the
// exact fallback: 8-bit radix rounds over the whole key with per-warp
// histograms over contiguous warp slices, then an emit pass taking threshold
// ties in token-id order.
#include "dt_launch.h"
#include "kn1_common.cuh"

namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int UNR = 4;      // vectors per step of pass 1; loads in flight per thread in pass 2
constexpr int RING = 8;     // per-thread ring of 16-byte vectors in pass 1 (two CTAs per SM)
constexpr int RING_DEEP = 16;  // the same when every row has an SM to itself: more bytes in flight
constexpr int CAP = 2048;   // candidates of a row

struct Kn1bMisc {
    float wm[NW];  // per-warp running maximum and sum
    float ws[NW];
    float m;       // row maximum
    float lse;
    int ncand;
    int nsel;
    int nslot;     // slots whose maximum reaches the bound (short lists)
    int outside;   // counting rank: an entry lies outside the 256 buckets
    int weq[NW];   // fallback: threshold ties per warp slice
    int red[NW];   // block scans
    DtBinSearch bs;
};

// Dynamic shared memory: [misc 1 KB][hist 1 KB][rank scratch 4 KB][cand CAP*8]
// [work CAP*8][extra 11 KB][ring RING*NT*16].  Ring slot k of thread t sits at
// (k * NT + t) * 16 bytes, so a warp's 16-byte reads of one slot are
// conflict-free.  Areas change roles along a row: cand + work + extra hold
// the groups' 16-bit maximum words (KEYCAP of them) from pass 1 until the
// listing; the ring, once pass 1 is done, holds the list of groups and the
// staged re-reads until pass 2 ends, then the counting rank's per-entry
// offsets; cand holds the candidates from pass 2 on; work holds the rank's
// per-warp histograms or buckets, or the fallback's per-warp histograms (NW
// KB).  The extra area fills the shared memory that two CTAs per SM leave.
constexpr size_t OFF_HIST = 1024;
constexpr size_t OFF_RS = OFF_HIST + 1024;
constexpr size_t OFF_CAND = OFF_RS + 4096;
constexpr size_t OFF_WORK = OFF_CAND + (size_t)CAP * 8;
constexpr size_t OFF_RING = OFF_WORK + (size_t)CAP * 8 + 11 * 1024;
constexpr int KEYCAP = (int)((OFF_RING - OFF_CAND) / 2);  // 16-bit group words
constexpr int C8MAX = (KEYCAP / NT + 7) / 8;               // 16-byte word reads per thread, at most
constexpr int P2RUN = 4;                                   // pass 2: items per thread and round, at most
// Candidate lists longer than this take the per-vector words; shorter ones
// re-read whole slots (a few times Kc x 9 vectors at V = 151936), which costs
// less than writing a word per vector in pass 1.
constexpr int KC_WORDS = 128;
template <int R>
constexpr size_t smem_of() { return OFF_RING + (size_t)R * NT * 16; }
constexpr size_t SMEM = smem_of<RING>();
static_assert(2 * (SMEM + 1024) <= 233472, "two CTAs per SM with the shallow ring");
static_assert(smem_of<RING_DEEP>() + 1024 <= 233472, "one CTA per SM with the deep ring");
static_assert(sizeof(Kn1bMisc) <= OFF_HIST, "misc block overflows its slot");
static_assert(sizeof(DtRankScratch) <= 4096, "rank scratch overflows its slot");
static_assert((size_t)CAP * 8 >= (size_t)NW * 1024, "per-warp histograms must fit the work area");
static_assert(C8MAX * 8 <= 64, "a thread's listing flags fit 64 bits");
static_assert((size_t)KEYCAP * 2 + 16 * 1024 <= (size_t)RING * NT * 16,
              "the group list and a stage of 1024 vectors must fit the ring");
static_assert((size_t)CAP * 2 <= (size_t)RING * NT * 16, "the rank offsets must fit the ring");
static_assert(NT * UNR * 4 <= CAP * 8, "the slot list must fit the work area");

template <typename T>
DT_DI uint4 ldv(const T* row, int v) {
    return __ldg(reinterpret_cast<const uint4*>(row) + v);
}


// (M, S) <- the merge of two running (max, sum) pairs.
DT_DI void merge_pair(float& M, float& S, float M2, float S2) {
    const float NEG_INF = -__int_as_float(0x7F800000);
    const float log2e = 1.44269504088896340736f;
    const float Mn = fmaxf(M, M2);
    const float a = (M == NEG_INF) ? 0.f : __fmul_rn(S, dt_ex2_approx(__fmul_rn(__fsub_rn(M, Mn), log2e)));
    const float b = (M2 == NEG_INF) ? 0.f : __fmul_rn(S2, dt_ex2_approx(__fmul_rn(__fsub_rn(M2, Mn), log2e)));
    M = Mn;
    S = __fadd_rn(a, b);
}

// Exact fallback for a row whose candidates overflowed the buffer: 8-bit radix
// rounds over the whole key, per-warp histograms over contiguous warp slices,
// then an emit pass that takes threshold ties in token-id order; the Kc
// selected are ranked and written.  Kept out of line so that its registers do
// not weigh on the common path.
template <typename T>
__device__ __noinline__ void fallback_row(const T* __restrict__ rp, int V, int nfull, int nvec, int Kc, float lse,
                                          uint32_t mk16, int row, Kn1bMisc* misc, uint32_t* hist, DtRankScratch* rs,
                                          unsigned long long* cand, unsigned char* work,
                                          int32_t* __restrict__ cand_id, float* __restrict__ cand_lp) {
    using E = DtElem<T>;
    constexpr int EPV = 16 / sizeof(T);
    const float NEG_INF = -__int_as_float(0x7F800000);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t* whist = (uint32_t*)work;
    unsigned long long* bucket = (unsigned long long*)work;
    // ---- fallback: exact radix select over the whole key --------------
    const int vseg = (nvec + NW - 1) / NW;
    const int v0 = min(nvec, wid * vseg), v1 = min(nvec, v0 + vseg);
    uint32_t* myh = whist + wid * 256;
    auto get = [&](int v, float (&x)[EPV]) {  // values, -inf past the row
        if (v < nfull) {
            dt_vec_vals<T>(ldv(rp, v), x);
        } else {
#pragma unroll
            for (int s = 0; s < EPV; ++s) x[s] = v * EPV + s < V ? E::val(rp[v * EPV + s]) : NEG_INF;
        }
    };
    uint32_t T_key = 0;
    int need = Kc, last_bin = 0;
    for (int rd = 0; rd < E::KB / 8; ++rd) {
        const int shift = E::KB - 8 - 8 * rd;
        const uint32_t pre = rd ? (T_key >> (shift + 8)) : 0u;
        __syncthreads();
        for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
        __syncthreads();
        for (int v = v0 + lane; v < v1; v += 32) {
            float x[EPV];
            get(v, x);
#pragma unroll
            for (int s = 0; s < EPV; ++s) {
                const uint32_t k = E::key(dt_to_elem<T>(x[s]));
                if (v * EPV + s < V && (rd == 0 || (k >> (shift + 8)) == pre))
                    atomicAdd(&myh[(k >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t a = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
            hist[tid] = a;
        }
        __syncthreads();
        dt_find_bin<true>(hist, need, &misc->bs);
        const uint32_t dg = (uint32_t)misc->bs.digit;
        need = misc->bs.need;
        T_key |= dg << shift;
        last_bin = (int)dg;
    }
    // threshold ties per warp slice, from the last round's histograms
    if (tid < NW) misc->weq[tid] = (int)whist[tid * 256 + last_bin];
    __syncthreads();
    int eqbase = 0;
    for (int w = 0; w < wid; ++w) eqbase += misc->weq[w];
    const float Tv = E::key_val(T_key);
    int running = 0;
    for (int base = v0; base < v1; base += 32) {
        const int v = base + lane;
        float x[EPV];
        int neq = 0;
        if (v < v1) {
            get(v, x);
#pragma unroll
            for (int s = 0; s < EPV; ++s) neq += (v * EPV + s < V && x[s] == Tv);
        }
        const int inc = dt_warp_incl_scan(neq);
        int r = running + inc - neq;  // ties before this lane's vector in this warp slice
        running += __shfl_sync(0xffffffffu, inc, 31);
        if (v < v1) {
#pragma unroll
            for (int s = 0; s < EPV; ++s) {
                if (v * EPV + s >= V || !(x[s] >= Tv)) continue;
                bool take = true;
                if (x[s] == Tv) {
                    take = (eqbase + r < need);
                    ++r;
                }
                if (take) {
                    const int slot = atomicAdd(&misc->nsel, 1);
                    if (slot < Kc)
                        cand[slot] = ((unsigned long long)E::key(dt_to_elem<T>(x[s])) << 32) |
                                     (unsigned long long)(0xFFFFFFFFu - (uint32_t)(v * EPV + s));
                }
            }
        }
    }
    __syncthreads();
    const int tot = min(misc->nsel, Kc);
    // the per-warp histograms are no longer read: `work` becomes the buckets
    if (tot <= 64 ||
        !dt_bucket_rank_and_write<T, NT>(cand, tot, 0, tot, mk16, Kc, lse, row, cand_id, cand_lp, rs,
                                         bucket)) {
        if (tot <= 64) dt_rank_and_write<T, NT>(cand, tot, cand, tot, Kc, lse, row, cand_id, cand_lp);
        else dt_sort_and_write<T, NT>(cand, tot, Kc, 0, 1, lse, row, cand_id, cand_lp);
    }
}

// The 16-bit word a group leaves for its maximum x: bf16 keeps the raw bits
// (one shift; compared later as values), fp32 the top 16 bits of the
// order key (truncating the raw bits would misorder tiny negatives).
template <typename T> DT_DI uint16_t group_word(float x);
template <> DT_DI uint16_t group_word<uint16_t>(float x) { return (uint16_t)(__float_as_uint(x) >> 16); }
template <> DT_DI uint16_t group_word<float>(float x) { return (uint16_t)(DtElem<float>::key(x) >> 16); }
// Bits e = 0..7: does word e of the 16-byte read w reach the bound?  bf16
// compares the raw words as values, two per instruction (a NaN word never
// reaches); fp32 compares the key words with b16.
template <typename T> DT_DI uint32_t reach8(const uint4& w, float bound, uint32_t b16);
template <> DT_DI uint32_t reach8<uint16_t>(const uint4& w, float bound, uint32_t) {
    const __nv_bfloat162 th = __float2bfloat162_rn(bound);  // exact: the bound is a bf16 value
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t f = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t m = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&ww[i]), th);
        f |= ((m & 1u) | ((m >> 15) & 2u)) << (2 * i);
    }
    return f;
}
template <> DT_DI uint32_t reach8<float>(const uint4& w, float, uint32_t b16) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t f = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        f |= ((uint32_t)((ww[i] & 0xFFFFu) >= b16) | ((uint32_t)((ww[i] >> 16) >= b16) << 1)) << (2 * i);
    return f;
}
// The word of a group that holds no vector: a NaN for bf16, which reaches no
// bound; key 0 for fp32, which reaches only the -inf bound (whose re-read
// then finds no vector to load).
template <typename T> DT_DI uint16_t group_none();
template <> DT_DI uint16_t group_none<uint16_t>() { return 0xFFFFu; }
template <> DT_DI uint16_t group_none<float>() { return 0u; }

// Rank the row's `total` candidates (bf16 entries in token-id order) by a
// stable counting sort on their value: bucket b = mk16 - key holds one bf16
// value (b = 0: the row maximum), so an entry's rank is the number of entries
// in earlier buckets plus those of its own bucket listed before it.  Each warp
// counts a contiguous slice of the list (peers found with ballots);
// a column scan of the per-warp histograms then gives every (warp, bucket) its
// first rank.  Entries of rank < Kc are written.  Returns false, having
// written nothing, when an entry lies 256 or more values below the maximum
// (the caller sorts instead).  Block-uniform; contains __syncthreads.
DT_DI bool counting_rank_bf16(const unsigned long long* cand, int total, uint32_t mk16, int Kc, float lse, int row,
                              int32_t* __restrict__ cand_id, float* __restrict__ cand_lp, uint32_t* whist,
                              uint16_t* loc, Kn1bMisc* misc) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
    if (tid == 0) misc->outside = 0;
    __syncthreads();
    const int per = ((total + NW * 32 - 1) / (NW * 32)) * 32;  // entries per warp, a multiple of 32
    const int lo = min(total, wid * per), hi = min(total, lo + per);
    uint32_t* mine = whist + wid * 256;
    for (int c0 = lo; c0 < hi; c0 += 32) {  // warp-uniform trip count
        const int i = c0 + lane;
        uint32_t b = 0x10000u + (uint32_t)lane;  // a lane past the slice matches no other
        if (i < hi) {
            const uint32_t bi = mk16 - (uint32_t)(cand[i] >> 32);
            if (bi < 256u) b = bi;
            else misc->outside = 1;
        }
        // lanes with the same bucket: eight ballots on its bits (a valid lane's
        // bucket is < 256, an idle lane's is not and it matches none)
        uint32_t peers = __ballot_sync(0xffffffffu, b < 256u);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t m = __ballot_sync(0xffffffffu, (b >> k) & 1u);
            peers &= ((b >> k) & 1u) ? m : ~m;
        }
        const uint32_t before = peers & ((1u << lane) - 1u);
        const uint32_t prior = b < 256u ? mine[b] : 0u;
        if (b < 256u) loc[i] = (uint16_t)(prior + __popc(before));
        __syncwarp();
        if (b < 256u && before == 0u) mine[b] = prior + __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    if (misc->outside) return false;
    // column scan: whist[w][b] <- first rank of warp w's entries in bucket b
    uint32_t sz = 0;
    if (tid < 256)
        for (int w = 0; w < NW; ++w) {
            const uint32_t c = whist[w * 256 + tid];
            whist[w * 256 + tid] = sz;
            sz += c;
        }
    int tot;
    const int start = dt_block_excl_scan<NT>(tid < 256 ? (int)sz : 0, misc->red, &tot);
    if (tid < 256)
        for (int w = 0; w < NW; ++w) whist[w * 256 + tid] += (uint32_t)start;
    __syncthreads();
    for (int i = tid; i < total; i += NT) {
        const unsigned long long e = cand[i];
        const int r = (int)(whist[(i / per) * 256 + (mk16 - (uint32_t)(e >> 32))] + loc[i]);
        if (r < Kc) dt_write_cand<uint16_t>(e, r, Kc, lse, row, cand_id, cand_lp);
    }
    return true;
}

// Bits 0..EPV-1: which elements of the 16-byte vector q reach the bound
// (bf16: two per packed compare; a NaN never reaches).
template <typename T> DT_DI uint32_t elem_bits(const uint4& q, float bound);
template <> DT_DI uint32_t elem_bits<uint16_t>(const uint4& q, float bound) { return reach8<uint16_t>(q, bound, 0); }
template <> DT_DI uint32_t elem_bits<float>(const uint4& q, float bound) {
    return (uint32_t)(__uint_as_float(q.x) >= bound) | ((uint32_t)(__uint_as_float(q.y) >= bound) << 1) |
           ((uint32_t)(__uint_as_float(q.z) >= bound) << 2) | ((uint32_t)(__uint_as_float(q.w) >= bound) << 3);
}

template <typename T, int RING>
__global__ void __launch_bounds__(NT, RING > 8 ? 1 : 2) kn1b_kernel(const T* __restrict__ logits, int V, int Kc, int rows,
                                                     float* __restrict__ lse_out, int32_t* __restrict__ cand_id,
                                                     float* __restrict__ cand_lp) {
    using E = DtElem<T>;
    constexpr int EPV = 16 / sizeof(T);
    const float NEG_INF = -__int_as_float(0x7F800000);
    extern __shared__ __align__(128) unsigned char smem[];
    Kn1bMisc* misc = (Kn1bMisc*)smem;
    uint32_t* hist = (uint32_t*)(smem + OFF_HIST);
    DtRankScratch* rs = (DtRankScratch*)(smem + OFF_RS);
    unsigned long long* cand = (unsigned long long*)(smem + OFF_CAND);
    uint16_t* keys = (uint16_t*)(smem + OFF_CAND);  // pass 1 .. listing: cand + work + extra
    uint16_t* list = (uint16_t*)(smem + OFF_RING);  // listing .. pass 2: the ring
    uint16_t* loc = (uint16_t*)(smem + OFF_RING);   // ranking: the ring
    unsigned long long* bucket = (unsigned long long*)(smem + OFF_WORK);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    // No early trigger: the rows fill the SMs' shared memory and the bandwidth, and blocks of the next
    // kernels parked beside them (waiting on this grid) only slowed the whole step down.
    dt_pdl_wait();  // the logits may come from the kernel just before us

    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        const T* rp = logits + (size_t)row * (size_t)V;
        const bool aligned = ((uintptr_t)rp & 15u) == 0;
        const int nfull = aligned ? V / EPV : 0;  // vectors read with 16-byte loads
        const int nvec = (V + EPV - 1) / EPV;
        // a group is GV consecutive vectors m of one thread (vector indices
        // NT apart): one vector unless the row is so long that the groups'
        // 16-bit words would not fit KEYCAP.  Word k = q * NT + t is thread
        // t's group q; with one vector per group k is the vector index itself.
        const int nmax = (nfull + NT - 1) / NT;  // most vectors of one thread
        int gshift = 0;
        while (((nmax + (1 << gshift) - 1) >> gshift) * NT > KEYCAP) ++gshift;
        const int GV = 1 << gshift;
        const int nq = (nmax + GV - 1) >> gshift;  // groups per thread, at most
        const bool words = Kc > KC_WORDS;  // block-uniform
        if (tid < 256) hist[tid] = 0;
        if (tid == 0) {
            misc->nsel = 0;
            misc->ncand = 0;
            misc->nslot = 0;
        }

        // ---- pass 1: running (max, sum exp), slot maxima, group words -------
        float M = NEG_INF, S = 0.f;
        // this thread's 16-byte vectors: m-th at vector index tid + m * NT
        const int nmine = nfull > tid ? (nfull - tid + NT - 1) / NT : 0;
        const int nqt = (nmine + GV - 1) >> gshift;  // this thread's groups
        // slot u: the thread's vectors m = u (mod UNR); their maxima bound the row's Kc-th logit
        float gm[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) gm[u] = NEG_INF;
        uint32_t gv = nmine >= UNR ? (1u << UNR) - 1 : (1u << nmine) - 1;  // bit u: slot u holds an element
        {
            // copies go in groups of two vectors, PRE groups ahead of use
            constexpr int G = 2, PRE = RING / G - 1;
            uint4* ring = (uint4*)(smem + OFF_RING) + tid;  // slot k at ring[k * NT]
            const uint4* src = reinterpret_cast<const uint4*>(rp) + tid;
            float grun = NEG_INF;  // maximum of the open group
            // vector m's maximum joins its group, whose word is rewritten with
            // the running maximum (no branch: the last write holds the group's)
            auto word = [&](int m, float vm) {
                grun = (m & (GV - 1)) ? fmaxf(grun, vm) : vm;
                keys[(m >> gshift) * NT + tid] = group_word<T>(grun);
            };
#pragma unroll
            for (int k = 0; k < PRE * G; ++k) {
                if (k < nmine) dt_cp_async16(ring + k * NT, src + (size_t)k * NT);
                if (k % G == G - 1) dt_cp_commit();
            }
            for (int m0 = 0; m0 < nmine; m0 += UNR) {
                const int rbase = m0 % RING;  // a multiple of UNR
#pragma unroll
                for (int h = 0; h < UNR / G; ++h) {
                    if (m0 + h * G < nmine) {
                        const int mi = m0 + (h + PRE) * G;  // first vector of the group to start
#pragma unroll
                        for (int j = 0; j < G; ++j)
                            if (mi + j < nmine)
                                dt_cp_async16(ring + ((rbase + (h + PRE) * G + j) % RING) * NT, src + (size_t)(mi + j) * NT);
                        dt_cp_commit();
                        dt_cp_wait<PRE>();  // this group has landed
                        // the group's two vectors fold into (M, S) together: one
                        // rescale check and two chains of packed adds per pair
                        static_assert(G == 2, "vectors are folded in pairs");
                        const int u = h * G;
                        if (m0 + u + 1 < nmine) {
                            const uint4 qa = ring[(rbase + u) * NT], qb = ring[(rbase + u + 1) * NT];
                            const float va = dt_vec_max<T>(qa), vb = dt_vec_max<T>(qb);
                            gm[u] = fmaxf(gm[u], va);
                            gm[u + 1] = fmaxf(gm[u + 1], vb);
                            if (words) {
                                word(m0 + u, va);
                                word(m0 + u + 1, vb);
                            }
                            float x[2 * EPV];
                            dt_vec_vals<T>(qa, *reinterpret_cast<float(*)[EPV]>(x));
                            dt_vec_vals<T>(qb, *reinterpret_cast<float(*)[EPV]>(x + EPV));
                            dt_online_add<2 * EPV>(x, fmaxf(va, vb), M, S);
                        } else {  // the thread's last vector, on its own
                            const uint4 q = ring[(rbase + u) * NT];
                            const float vm = dt_vec_max<T>(q);
                            gm[u] = fmaxf(gm[u], vm);
                            if (words) word(m0 + u, vm);
                            float x[EPV];
                            dt_vec_vals<T>(q, x);
                            dt_online_add<EPV>(x, vm, M, S);
                        }
                    }
                }
            }
            dt_cp_wait<0>();
        }
        // group rows the thread has no vectors in
        if (words)
            for (int q = nqt; q < nq; ++q) keys[q * NT + tid] = group_none<T>();
        // the rest -- a ragged last vector, or every vector of a row that is not
        // 16-byte aligned -- with element loads (-inf fill adds nothing)
        float tmax = NEG_INF;
        const bool has_tail = nfull + tid < nvec;
        for (int v = nfull + tid; v < nvec; v += NT) {
            float x[EPV];
            float vm = NEG_INF;
#pragma unroll
            for (int s = 0; s < EPV; ++s) {
                const int idx = v * EPV + s;
                x[s] = idx < V ? E::val(rp[idx]) : NEG_INF;
                vm = fmaxf(vm, x[s]);
            }
            tmax = fmaxf(tmax, vm);
            dt_online_add<EPV>(x, vm, M, S);
        }
        if (has_tail) {
            gm[0] = fmaxf(gm[0], tmax);
            gv |= 1u;
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
            const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
            merge_pair(M, S, M2, S2);
        }
        if (lane == 0) {
            misc->wm[wid] = M;
            misc->ws[wid] = S;
        }
        __syncthreads();
        if (wid == 0) {
            float m2 = lane < NW ? misc->wm[lane] : NEG_INF;
            float s2 = lane < NW ? misc->ws[lane] : 0.f;
            for (int o = 16; o > 0; o >>= 1) {
                const float M2 = __shfl_xor_sync(0xffffffffu, m2, o);
                const float S2 = __shfl_xor_sync(0xffffffffu, s2, o);
                merge_pair(m2, s2, M2, S2);
            }
            if (lane == 0) {
                misc->m = m2;
                misc->lse = m2 + logf(s2);
            }
        }
        __syncthreads();
        const float mrow = misc->m;
        const float lse = misc->lse;

        // ---- the bound: Kc-th largest slot maximum ---------------------------
        const uint32_t mk16 = E::key(dt_to_elem<T>(mrow)) >> (E::KB - 16);
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            if ((gv >> u) & 1u) {
                const uint32_t b = mk16 - (E::key(dt_to_elem<T>(gm[u])) >> (E::KB - 16));
                if (b < 256u) atomicAdd(&hist[b], 1u);
            }
        }
        __syncthreads();
        dt_find_bin<false>(hist, Kc, &misc->bs);
        float bound = NEG_INF;
        uint32_t b16 = 0;  // a group reaches the bound iff its word's key is >= b16
        if (misc->bs.digit >= 0) {
            b16 = mk16 - (uint32_t)misc->bs.digit;
            // smallest value whose key has these top bits (keys <= 127 are -inf or NaN)
            if (b16 > 127u) bound = E::key_val(b16 << (E::KB - 16));
            else b16 = 0;
        }

        if (words) {
            // ---- list the groups that reach the bound in order of their word
            // index k: each thread takes a contiguous run of 8 * C8 words (16-byte
            // reads), one block scan orders the runs ----------------------------------
            const int nk = nq * NT;
            const int C8 = (nq + 7) >> 3;  // 16-byte reads per thread
            const uint4* kv = reinterpret_cast<const uint4*>(keys) + tid * C8;
            int nlist;
            {
                unsigned long long fm = 0;  // bit 8 r + e: word e of read r reaches the bound
                for (int r = 0; r < C8; ++r)
                    if ((tid * C8 + r) * 8 < nk) fm |= (unsigned long long)reach8<T>(kv[r], bound, b16) << (8 * r);
                int at = dt_block_excl_scan<NT>(__popcll(fm), misc->red, &nlist);
                while (fm) {
                    const int e = __ffsll(fm) - 1;
                    fm &= fm - 1;
                    list[at++] = (uint16_t)(tid * C8 * 8 + e);
                }
            }
            __syncthreads();  // the words are dead from here: cand, work and extra take new roles

            // ---- pass 2: re-read the listed groups, keep every element at or
            // above the bound ---------------------------------------------------------
            // item f: vector j = f mod GV of listed group f / GV.  With one vector
            // per group the item's vector is its list entry, so items run in
            // vector order and the candidates come out in token-id order.  Each
            // round stages up to `rcap` items in the ring after the list, every
            // thread a contiguous run of at most P2RUN, with asynchronous copies;
            // the thread reads back only its own run (no barrier), notes which
            // elements reach the bound, and a block scan places its candidates.
            const int nitems = nlist << gshift;
            uint4* stage = (uint4*)(smem + OFF_RING + (((size_t)nlist * 2 + 15) & ~(size_t)15));
            const int scap = (int)(((size_t)RING * NT * 16 - ((unsigned char*)stage - (smem + OFF_RING))) / 16);
            const int rcap = min(scap, P2RUN * NT);
            auto item_vec = [&](int f) {  // vector index of item f, nfull where there is none
                const int k = list[f >> gshift];
                const int v = (k & (NT - 1)) + (((k / NT) << gshift) + (f & (GV - 1))) * NT;
                return v < nfull ? v : nfull;
            };
            int ncand = 0;
            for (int r0 = 0; r0 < nitems; r0 += rcap) {  // block-uniform trip count
                const int nr = min(rcap, nitems - r0);
                const int cpt = (nr + NT - 1) / NT;
                const int s0 = tid * cpt, s1 = min(nr, s0 + cpt);  // this thread's run, within the round
                for (int k = s0; k < s1; ++k) {
                    const int v = item_vec(r0 + k);
                    if (v < nfull) dt_cp_async16(stage + k, reinterpret_cast<const uint4*>(rp) + v);
                }
                dt_cp_commit();
                dt_cp_wait<0>();
                uint32_t bits = 0;  // bit EPV * (k - s0) + e: element e of item k reaches the bound
                for (int k = s0; k < s1; ++k)
                    if (item_vec(r0 + k) < nfull) bits |= elem_bits<T>(stage[k], bound) << (EPV * (k - s0));
                int tot;
                int w = ncand + dt_block_excl_scan<NT>(__popc(bits), misc->red, &tot);
                while (bits) {
                    const int bi = __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int k = s0 + bi / EPV, e = bi % EPV;
                    if (w < CAP) {
                        const T xe = reinterpret_cast<const T*>(stage + k)[e];
                        cand[w] = ((unsigned long long)E::key(xe) << 32) |
                                  (unsigned long long)(0xFFFFFFFFu - (uint32_t)(item_vec(r0 + k) * EPV + e));
                    }
                    ++w;
                }
                ncand += tot;
                __syncthreads();  // the stage is reused by the next round
            }
            if (tid == 0) misc->ncand = ncand;
            __syncthreads();
        } else {
            // ---- pass 2, short lists: re-read the slots that reach the bound
            // (each of its vectors UNR * NT apart); unordered
            auto keep = [&](float xv, int idx) {
                const int slot = atomicAdd(&misc->ncand, 1);
                if (slot < CAP)
                    cand[slot] = ((unsigned long long)E::key(dt_to_elem<T>(xv)) << 32) |
                                 (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
            };
            int* slots = (int*)(smem + OFF_WORK);
#pragma unroll
            for (int u = 0; u < UNR; ++u)
                if (((gv >> u) & 1u) && gm[u] >= bound && tid + u * NT < nfull)
                    slots[atomicAdd(&misc->nslot, 1)] = tid + u * NT;  // first vector of the slot
            __syncthreads();
            // a slot's vectors are UNR * NT apart, per of them; a warp takes spw
            // listed slots at a time, lane = (slot dj, vector kc + k), kl
            // vectors of a slot per pass
            const int per = (nfull + UNR * NT - 1) / (UNR * NT);
            const int kl = per < 32 ? per : 32;
            const int spw = kl > 0 ? 32 / kl : 1;
            const int dj = kl > 0 ? lane / kl : 0, k = kl > 0 ? lane % kl : 0;
            const int nslot = misc->nslot;
            for (int kc = 0; kc < per; kc += kl) {
                for (int j0 = wid * spw; j0 < nslot; j0 += 2 * NW * spw) {
                    uint4 q[2];
                    int vv[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = j0 + h * NW * spw + dj;
                        vv[h] = (dj < spw && j < nslot && kc + k < per) ? slots[j] + (kc + k) * (UNR * NT) : nfull;
                        if (vv[h] < nfull) q[h] = ldv(rp, vv[h]);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (vv[h] < nfull && dt_vec_max<T>(q[h]) >= bound) {
                            float x[EPV];
                            dt_vec_vals<T>(q[h], x);
#pragma unroll
                            for (int e = 0; e < EPV; ++e)
                                if (x[e] >= bound) keep(x[e], vv[h] * EPV + e);
                        }
                    }
                }
            }
            __syncthreads();
        }
        // the element-loaded rest, unordered
        if (has_tail && tmax >= bound) {
            for (int v = nfull + tid; v < nvec; v += NT) {
#pragma unroll
                for (int s = 0; s < EPV; ++s) {
                    const int idx = v * EPV + s;
                    if (idx < V) {
                        const float xv = E::val(rp[idx]);
                        if (xv >= bound) {
                            const int slot = atomicAdd(&misc->ncand, 1);
                            if (slot < CAP)
                                cand[slot] = ((unsigned long long)E::key(dt_to_elem<T>(xv)) << 32) |
                                             (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
                        }
                    }
                }
            }
        }
        __syncthreads();
        const int total = misc->ncand;

        if (total <= CAP) {
            bool done = false;
            if (sizeof(T) == 2 && words && nvec == nfull && GV == 1 && total > 128)  // bf16, in token-id order
                done = counting_rank_bf16(cand, total, mk16, Kc, lse, row, cand_id, cand_lp, (uint32_t*)(smem + OFF_WORK),
                                          loc, misc);
            if (!done) {
                if (total <= 128) {
                    dt_rank16_and_write<T, NT>(cand, total, cand, total, Kc, lse, row, cand_id, cand_lp);
                } else if (!dt_bucket_rank_and_write<T, NT>(cand, total, 0, total, mk16, Kc, lse, row, cand_id,
                                                            cand_lp, rs, bucket)) {
                    dt_sort_and_write<T, NT>(cand, total, Kc, 0, 1, lse, row, cand_id, cand_lp);
                }
            }
        } else {
            fallback_row<T>(rp, V, nfull, nvec, Kc, lse, mk16, row, misc, hist, rs, cand, smem + OFF_WORK, cand_id,
                            cand_lp);
        }
        if (tid == 0) lse_out[row] = lse;
        __syncthreads();  // the next row reuses every buffer
    }
}

}  // namespace

size_t dt_kn1b_smem_bytes() { return SMEM; }

template <typename T, int R>
cudaError_t kn1b_launch_t(const void* logits, int rows, int V, int Kc, float* lse, int32_t* cand_id, float* cand_lp,
                          cudaStream_t st) {
    constexpr size_t sm = smem_of<R>();
    cudaError_t e = cudaFuncSetAttribute(kn1b_kernel<T, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    DtLaunch lc(dim3(rows, 1, 1), dim3(NT, 1, 1), sm, st);
    return cudaLaunchKernelEx(&lc.cfg, kn1b_kernel<T, R>, (const T*)logits, V, Kc, rows, lse, cand_id, cand_lp);
}

cudaError_t dt_kn1b_launch(const void* logits, int dtype, int rows, int V, int Kc, float* lse, int32_t* cand_id,
                           float* cand_lp, cudaStream_t st) {
    // rows that each get an SM to themselves stream with the deep ring
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess) {
            (void)cudaGetLastError();
            sms = -1;
        }
    }
    const bool deep = sms > 0 && rows <= sms;
    if (dtype == DT_BF16)
        return deep ? kn1b_launch_t<uint16_t, RING_DEEP>(logits, rows, V, Kc, lse, cand_id, cand_lp, st)
                    : kn1b_launch_t<uint16_t, RING>(logits, rows, V, Kc, lse, cand_id, cand_lp, st);
    return deep ? kn1b_launch_t<float, RING_DEEP>(logits, rows, V, Kc, lse, cand_id, cand_lp, st)
                : kn1b_launch_t<float, RING>(logits, rows, V, Kc, lse, cand_id, cand_lp, st);
}
