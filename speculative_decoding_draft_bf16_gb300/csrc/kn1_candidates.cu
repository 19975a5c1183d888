// kn1_candidates.cu -- stage 1: per-position log-softmax and exact Top-Kc.
//
// [DARTree] Algorithm 1, its per-position Top-K candidate step; [DDTree] section 3.3
// (log-domain scores of each position's Top-K tokens).
//
// One thread-block cluster of S CTAs per row (request b, position l); CTA c
// owns a contiguous vocabulary chunk, staged once from HBM into shared memory
// by a 1-D bulk async copy and then read 16 bytes per lane at a time.
//
// Fast path (two cluster barriers per row):
//   pass 1   each lane's running maximum and sum exp(x - max) over its
//            elements (rescaled whenever the maximum grows); the lane maxima
//            (one per thread) go into a 256-bin histogram of order keys below
//            the chunk maximum; the lanes' (max, sum) pairs merge into the
//            chunk's;
//   barrier  1;
//   exchange every lane maximum is a distinct element of the row, so the
//            Kc-th largest lane maximum of the row is a lower bound for its
//            Kc-th largest logit.  Every CTA merges the cluster's histograms
//            in the frame of the row maximum through DSMEM (entries that fall
//            outside the frame are dropped, which can only lower the bound)
//            and reads the bound off the top, and merges the chunks' (max,
//            sum) pairs into the row's normaliser;
//   pass 2   collect every element at or above the bound as a candidate (a
//            vector is looked into only when its maximum reaches the bound);
//            then every CTA appends its candidates to every CTA's row list
//            (one remote atomic per destination for the offset, then plain
//            remote stores);
//   barrier  2;
//   rank     each CTA now holds the row's whole candidate list locally and
//            ranks its own candidates in it (logit descending, token id
//            ascending), writing those of rank < Kc.  No shared memory of
//            another CTA is touched after the second barrier.
// Rows whose candidates overflow the buffers (a row of many equal logits, a
// tiny vocabulary) take the fallback, the same for the whole cluster: a 256-bin
// window histogram of all keys below the chunk maximum, the exact threshold
// found across the cluster (fp32: two more radix rounds; a window holding
// fewer than Kc keys: full radix from the top), threshold ties taken in
// token-id order.
// Every logit is read from HBM once.  A row whose staging wait ran out of its
// bound gets a NaN normaliser (the selection kernels turn that into
// DT_DEV_TIMEOUT).
#include "dt_launch.h"
#include "kn1_common.cuh"

namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int SMAX = 16;
constexpr int CCAP = 1024;  // candidates one CTA keeps (>= the largest Kc)
constexpr int ACAP = 2048;  // candidates of one row

// Per-row values of the fallback that partners read after its cluster
// barriers, kept per row parity: a CTA may start its next row while a partner
// still reads them.
struct RowPub {
    int ncand;    // candidates found in this CTA (may exceed CCAP)
    int nsel;     // fallback: selected entries in this CTA
};

// Values partners read between a row's two barriers are written before the
// first and not again before the second has passed, so they need no parity.
// A CTA's per-row statistics, pushed into every CTA of the cluster.
struct Kn1Stat {
    float m;        // chunk max value
    float s;        // chunk sum exp(x - m)
    uint32_t mk16;  // chunk max key, top 16 bits
    int timeout;    // the chunk's staging wait ran out
};

struct Kn1Misc {
    uint64_t bar;      // the chunk copy
    uint64_t probe;    // the timeout-path test hook's barrier (never completes)
    int timeout;       // this row: this CTA's staging wait ran out
    int nrecv;         // this row: candidates the cluster has appended to `all`
    RowPub pub[2];
    Kn1Stat pin[SMAX]; // this row: every CTA's statistics, pushed by each before the first barrier
    uint32_t cmk[SMAX];
    int pbase[SMAX];   // this CTA's offset in each partner's list
    int ceq[SMAX];
    int cnsel[SMAX];
    float lse;
    DtBinSearch bs;
    int weq[NW];       // fallback: threshold ties per warp slice
    float red_f[NW];   // per-warp maxima
    float red_s[NW];   // per-warp sums
};

// Dynamic shared memory: [misc 1 KB][chist 2 KB][cand CCAP*8][all ACAP*8]
// [hin SMAX*1 KB][chunk data + 32].  The fallback's per-warp histograms
// (NW*1 KB) live in `all`, which it fills only after its last histogram read.
// hin[j] receives CTA j's lane-maximum histogram (its own frame) each row.
constexpr size_t OFF_CHIST = 1024;
constexpr size_t OFF_CAND = OFF_CHIST + 2048;
constexpr size_t OFF_ALL = OFF_CAND + (size_t)CCAP * 8;
constexpr size_t OFF_HIN = OFF_ALL + (size_t)ACAP * 8;
constexpr size_t OFF_DATA = OFF_HIN + (size_t)SMAX * 1024;
static_assert((size_t)ACAP * 8 >= (size_t)NW * 1024, "per-warp histograms must fit in the gather buffer");
static_assert(sizeof(Kn1Misc) <= OFF_CHIST, "misc block overflows its slot");
static_assert(OFF_DATA % 128 == 0, "chunk data must stay 128-byte aligned");

// Vector access to the staged chunk: vector j (16 bytes) holds elements
// j*EPV - h .. j*EPV - h + EPV - 1, where h is the head misalignment.
template <typename T>
struct Chunk {
    static constexpr int EPV = 16 / sizeof(T);
    const uint4* v;  // 16-byte aligned base
    int h;           // elements of vector 0 that precede the chunk
    int n;           // elements in the chunk
    int nv;          // vectors covering the chunk
    DT_DI void unpack(const uint4& q, T (&e)[EPV]) const {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                e[2 * k] = (T)(w[k] & 0xFFFFu);
                e[2 * k + 1] = (T)(w[k] >> 16);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) e[k] = __uint_as_float(w[k]);
        }
    }
};

// Warp w owns vectors [w*vseg, min(nv, (w+1)*vseg)).
DT_DI void warp_vectors(int nv, int* v0, int* v1) {
    const int w = threadIdx.x >> 5;
    const int vseg = (nv + NW - 1) / NW;
    *v0 = min(nv, w * vseg);
    *v1 = min(nv, *v0 + vseg);
}

// g[t] = sum over the cluster's CTAs j of their 256-bin histogram `h` (each
// in its own frame: bin i counts keys with top bits refs[j] - i), re-framed
// at `top` (bin t counts keys with top bits top - t).  Entries outside the new
// frame are dropped.  Ends with __syncthreads.
DT_DI void merge_framed(cg::cluster_group& cluster, const uint32_t* h, int S, const uint32_t* refs, uint32_t top,
                        uint32_t* g) {
    const int t = threadIdx.x;
    if (t < 256) {
        uint32_t part[SMAX];
#pragma unroll
        for (int j = 0; j < SMAX; ++j) {
            part[j] = 0;
            const int wj = t - (int)(top - refs[j < S ? j : 0]);
            if (j < S && wj >= 0 && wj < 256) part[j] = cluster.map_shared_rank(h, j)[wj];
        }
        uint32_t a = 0;
#pragma unroll
        for (int j = 0; j < SMAX; ++j) a += part[j];
        g[t] = a;
    }
    __syncthreads();
}

// The same from histograms already copied into this CTA (hin[j]: CTA j's).
DT_DI void merge_framed_local(const uint32_t* hin, int S, const uint32_t* refs, uint32_t top, uint32_t* g) {
    const int t = threadIdx.x;
    if (t < 256) {
        uint32_t a = 0;
        for (int j = 0; j < S; ++j) {
            const int wj = t - (int)(top - refs[j]);
            if (wj >= 0 && wj < 256) a += hin[j * 256 + wj];
        }
        g[t] = a;
    }
    __syncthreads();
}

// Sum over the cluster of bin-aligned histograms (buffer `h` of every CTA).
DT_DI void merge_plain(cg::cluster_group& cluster, const uint32_t* h, int S, uint32_t* g) {
    const int t = threadIdx.x;
    if (t < 256) {
        uint32_t part[SMAX];
#pragma unroll
        for (int j = 0; j < SMAX; ++j) part[j] = (j < S) ? cluster.map_shared_rank(h, j)[t] : 0u;
        uint32_t a = 0;
#pragma unroll
        for (int j = 0; j < SMAX; ++j) a += part[j];
        g[t] = a;
    }
    __syncthreads();
}

// Probe budget of the timeout-path test hook (0: off), set by dt_kn1_set_probe.
__device__ long long g_kn1_probe;

// One CTA per SM: the registers this allows keep the fast path free of
// spills, and a CTA never shares its SM with a partner of the same row pass
// (the cluster size is chosen so that every row's cluster fits at once).
template <typename T>
__global__ void __launch_bounds__(NT, 1) kn1_kernel(const T* __restrict__ logits, int V, int chunk, int Kc, int rows,
                                                 float* __restrict__ lse_out,
                                                 int32_t* __restrict__ cand_id,
                                                 float* __restrict__ cand_lp) {
    using E = DtElem<T>;
    constexpr int EPV = Chunk<T>::EPV;
    const float NEG_INF = -__int_as_float(0x7F800000);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t g[256];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int c = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int lo = min(V, c * chunk), hi = min(V, lo + chunk);
    const int G = gridDim.y;  // clusters; cluster q takes rows q, q + G, q + 2G, ...

    Kn1Misc* misc = (Kn1Misc*)smem;
    uint32_t* chist = (uint32_t*)(smem + OFF_CHIST);
    unsigned long long* cand = (unsigned long long*)(smem + OFF_CAND);
    unsigned long long* all = (unsigned long long*)(smem + OFF_ALL);
    uint32_t* hin = (uint32_t*)(smem + OFF_HIN);

    if (tid == 0) {
        dt_mbar_init(&misc->bar, 1);
        dt_mbar_init(&misc->probe, 1);
        dt_fence_mbar_init();
    }
    dt_pdl_trigger();
    __syncthreads();
    dt_pdl_wait();  // the logits may come from the kernel just before us

    // chunk buffers (bit i of a mask: buffer i): a bulk copy not yet waited
    // for, and the parity of the buffer's next mbarrier completion
    // the chunk copy: pending (issued, not waited for) and its mbarrier phase
    bool pend = false;
    uint32_t phase = 0;
    DtStager<T> stg;  // ragged chunk ends of the copy, held in registers
    auto issue = [&](int r) {
        pend = stg.start(logits + (size_t)r * (size_t)V, lo, hi, smem + OFF_DATA, &misc->bar) != 0;
    };
    int row = blockIdx.y;
    if (row < rows) issue(row);

    bool fallback_taken = false;
    for (int it = 0; row < rows; ++it, row += G) {
        const int par = it & 1;
        const int nxt = row + G;
        RowPub* mp = &misc->pub[par];
        // partners stopped reading this CTA's per-row values at the previous
        // row's second barrier, and append to `all` only after the first
        if (tid == 0) {
            mp->ncand = 0;
            mp->nsel = 0;
            misc->timeout = 0;
            misc->nrecv = 0;
        }
        if (tid < 256) chist[tid] = 0;
        stg.finish(smem + OFF_DATA);  // this row's ragged ends
        // one thread waits on this row's copy; the others block in the barrier
        // below (blocked warps take no issue slots)
        if (pend) {
            if (tid == 0 && !dt_probe_wait(&misc->probe, g_kn1_probe)) misc->timeout = 1;
            if (tid == 0 && !dt_mbar_wait(&misc->bar, phase)) {
                misc->timeout = 1;
                dt_mbar_wait(&misc->bar, phase);
            }
            phase ^= 1u;
            pend = false;
        }
        __syncthreads();
        unsigned char* dbase = smem + OFF_DATA;
        Chunk<T> ch;
        // element lo sits at the source address's offset within 16 bytes
        ch.h = (int)(((uintptr_t)(logits + (size_t)row * (size_t)V + lo) & 15u) / sizeof(T));
        ch.v = (const uint4*)dbase;
        ch.n = hi - lo;
        ch.nv = (ch.h + ch.n + EPV - 1) / EPV;
        int v0, v1;
        warp_vectors(ch.nv, &v0, &v1);
        // vectors 0 and nv-1 may be partial (misaligned head, ragged tail);
        // they take the element-wise path
        const int full_lo = (ch.h > 0) ? 1 : 0;
        const int full_hi = ((ch.h + ch.n) % EPV == 0) ? ch.nv : ch.nv - 1;

        // ---- pass 1: lane maxima and running (max, sum exp) -----------------
        // two full vectors per step fold in together (one rescale check, two
        // chains of packed adds); partial vectors and a lone last one singly
        float lm = NEG_INF, ls = 0.f;
        auto fold1 = [&](int j) {
            const uint4 q = ch.v[j];
            float x[EPV];
            dt_vec_vals<T>(q, x);
            if (j >= full_lo && j < full_hi) {
                dt_online_add<EPV>(x, dt_vec_max<T>(q), lm, ls);
            } else {
                float vm = NEG_INF;
#pragma unroll
                for (int s = 0; s < EPV; ++s) {
                    const int idx = j * EPV + s - ch.h;
                    if (idx >= 0 && idx < ch.n) vm = fmaxf(vm, x[s]);
                    else x[s] = NEG_INF;
                }
                dt_online_add<EPV>(x, vm, lm, ls);
            }
        };
        {
            int j = v0 + lane;
            for (; j + 32 < v1; j += 64) {
                if (j >= full_lo && j + 32 < full_hi) {
                    const uint4 qa = ch.v[j], qb = ch.v[j + 32];
                    float x[2 * EPV];
                    dt_vec_vals<T>(qa, *reinterpret_cast<float(*)[EPV]>(x));
                    dt_vec_vals<T>(qb, *reinterpret_cast<float(*)[EPV]>(x + EPV));
                    dt_online_add<2 * EPV>(x, fmaxf(dt_vec_max<T>(qa), dt_vec_max<T>(qb)), lm, ls);
                } else {
                    fold1(j);
                    fold1(j + 32);
                }
            }
            if (j < v1) fold1(j);
        }
        const bool has = v0 + lane < v1;  // every vector holds at least one element
        // the chunk maximum first; then every lane scales its sum to it (one
        // exponential per lane, all in parallel) and the sums are plain adds
        const float wmax = dt_warp_max(lm);
        if (lane == 0) misc->red_f[wid] = wmax;
        __syncthreads();
        float m_c = NEG_INF;
#pragma unroll
        for (int w = 0; w < NW; ++w) m_c = fmaxf(m_c, misc->red_f[w]);
        const float log2e = 1.44269504088896340736f;
        const float scaled = (lm == NEG_INF) ? 0.f : __fmul_rn(ls, dt_ex2_approx(__fmul_rn(__fsub_rn(lm, m_c), log2e)));
        const float wsum = dt_warp_sum(scaled);
        if (lane == 0) misc->red_s[wid] = wsum;
        const bool any = ch.n > 0;
        const uint32_t mk16 = any ? (E::key(dt_to_elem<T>(m_c)) >> (E::KB - 16)) : 0u;
        {
            // lane maxima into the histogram: one atomic per distinct bin of a warp
            const uint32_t bn = has ? mk16 - (E::key(dt_to_elem<T>(lm)) >> (E::KB - 16)) : 0xFFFFFFFFu;
            const uint32_t same = __match_any_sync(0xffffffffu, bn);
            if (bn < 256u && lane == __ffs(same) - 1) atomicAdd(&chist[bn], (uint32_t)__popc(same));
        }
        __syncthreads();  // red_s and the histogram are complete
        if (tid < S) {
            // the chunk's (max, sum) with the timeout flag, pushed to every CTA
            float cs = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) cs += misc->red_s[w];
            *cluster.map_shared_rank(&misc->pin[c], tid) = Kn1Stat{m_c, cs, mk16, misc->timeout};
        }
        // push the histogram into slot c of every CTA's hin
        for (int i = tid; i < S * 256; i += NT) cluster.map_shared_rank(hin, i >> 8)[c * 256 + (i & 255)] = chist[i & 255];
        cluster.sync();  // barrier 1: every CTA holds every CTA's statistics and histogram

        // ---- exchange (local): the bound from the lane maxima; the row's normaliser
        if (tid < S) misc->cmk[tid] = misc->pin[tid].mk16;
        __syncthreads();
        uint32_t Mk16 = 0;
        for (int j = 0; j < S; ++j) Mk16 = max(Mk16, misc->cmk[j]);
        merge_framed_local(hin, S, misc->cmk, Mk16, g);
        dt_find_bin<false>(g, Kc, &misc->bs);
        float bound = NEG_INF;
        if (misc->bs.digit >= 0) {
            const uint32_t b16 = Mk16 - (uint32_t)misc->bs.digit;
            // smallest value whose key has these top bits (keys <= 127 are -inf or NaN)
            if (b16 > 127u) bound = E::key_val(b16 << (E::KB - 16));
        }
        if (tid == 0) {
            float M = misc->pin[0].m;
            for (int j = 1; j < S; ++j) M = fmaxf(M, misc->pin[j].m);
            float ssum = 0.f;
            for (int j = 0; j < S; ++j)
                if (misc->pin[j].m != NEG_INF) ssum += misc->pin[j].s * __expf(misc->pin[j].m - M);
            misc->lse = M + logf(ssum);
        }

        // ---- pass 2: candidates at or above the bound -----------------------
        for (int j = v0 + lane; j < v1; j += 32) {
            const uint4 q = ch.v[j];
            float x[EPV];
            if (j >= full_lo && j < full_hi) {
                if (dt_vec_max<T>(q) >= bound) {
                    dt_vec_vals<T>(q, x);
#pragma unroll
                    for (int s = 0; s < EPV; ++s) {
                        if (x[s] >= bound) {
                            const int slot = atomicAdd(&mp->ncand, 1);
                            if (slot < CCAP)
                                cand[slot] = ((unsigned long long)E::key(dt_to_elem<T>(x[s])) << 32) |
                                             (unsigned long long)(0xFFFFFFFFu - (uint32_t)(lo + j * EPV + s - ch.h));
                        }
                    }
                }
            } else {
                dt_vec_vals<T>(q, x);
#pragma unroll
                for (int s = 0; s < EPV; ++s) {
                    const int idx = j * EPV + s - ch.h;
                    if (idx >= 0 && idx < ch.n && x[s] >= bound) {
                        const int slot = atomicAdd(&mp->ncand, 1);
                        if (slot < CCAP)
                            cand[slot] = ((unsigned long long)E::key(dt_to_elem<T>(x[s])) << 32) |
                                         (unsigned long long)(0xFFFFFFFFu - (uint32_t)(lo + idx));
                    }
                }
            }
        }
        __syncthreads();
        // append this CTA's candidates to every CTA's row list; a CTA that found
        // more than it keeps adds a count that marks every list as overflowing
        const int nloc = mp->ncand;
        const int npush = nloc > CCAP ? 0 : nloc;
        if (tid < S) misc->pbase[tid] = atomicAdd(cluster.map_shared_rank(&misc->nrecv, tid), nloc > CCAP ? ACAP + 1 : nloc);
        __syncthreads();
        for (int i = tid; i < S * npush; i += NT) {
            const int d = i / npush, k = i - d * npush;
            const int at = misc->pbase[d] + k;
            if (at < ACAP) cluster.map_shared_rank(all, d)[at] = cand[k];
        }
        cluster.sync();  // barrier 2: every list complete

        // every CTA received every CTA's count, so the branch below is uniform
        // across the cluster (the fallback holds cluster barriers)
        const int total = misc->nrecv;
        const float lse = misc->lse;
        if (total <= ACAP) {
            if (total > DT_SORT_MIN) dt_sort_and_write<T, NT>(all, total, Kc, c, S, lse, row, cand_id, cand_lp);
            else dt_rank16_and_write<T, NT>(cand, nloc, all, total, Kc, lse, row, cand_id, cand_lp);
        } else {
            fallback_taken = true;
            // ---- fallback: window histogram over all keys, exact radix select
            uint32_t* whist = (uint32_t*)all;  // per-warp histograms
            uint32_t* myh = whist + wid * 256;
            for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
            __syncthreads();
            const uint32_t klo = mk16 >= 255u ? mk16 - 255u : 0u;
            const float x_lo = (klo <= 127u) ? NEG_INF : E::key_val(klo << (E::KB - 16));
            for (int j = v0 + lane; j < v1; j += 32) {
                float x[EPV];
                dt_vec_vals<T>(ch.v[j], x);
                const bool full = (j >= full_lo && j < full_hi);
#pragma unroll
                for (int s = 0; s < EPV; ++s) {
                    const int idx = j * EPV + s - ch.h;
                    if ((full || (idx >= 0 && idx < ch.n)) && x[s] >= x_lo)
                        atomicAdd(&myh[mk16 - (E::key(dt_to_elem<T>(x[s])) >> (E::KB - 16))], 1u);
                }
            }
            __syncthreads();
            // partners last read chist (the lane-maximum histogram) before the
            // previous cluster barrier, so it can be overwritten
            if (tid < 256) {
                uint32_t a = 0;
#pragma unroll
                for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
                chist[tid] = a;
            }
            __syncthreads();
            cluster.sync();
            merge_framed(cluster, chist, S, misc->cmk, Mk16, g);
            dt_find_bin<false>(g, Kc, &misc->bs);

            uint32_t T_key;
            int need;
            int cur = 0;        // chist buffer of the last round
            int last_bin = -1;  // per-warp histogram bin holding the threshold ties
            if (misc->bs.digit >= 0) {
                const uint32_t t16 = Mk16 - (uint32_t)misc->bs.digit;
                need = misc->bs.need;
                if (tid < S) {
                    const int wj = (int)(misc->cmk[tid] - t16);
                    misc->ceq[tid] = (wj >= 0 && wj < 256) ? (int)cluster.map_shared_rank(chist, tid)[wj] : 0;
                }
                last_bin = (int)(mk16 - t16);  // outside [0,256) when this CTA has no ties
                T_key = t16 << (E::KB - 16);
                if constexpr (E::KB == 32) {
                    // two radix rounds over the low 16 bits among keys with top bits t16
                    for (int rd = 0; rd < 2; ++rd) {
                        const int shift = 8 - 8 * rd;
                        const uint32_t pre = T_key >> (shift + 8);
                        __syncthreads();
                        for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
                        __syncthreads();
                        for (int j = v0 + lane; j < v1; j += 32) {
                            T e[EPV];
                            ch.unpack(ch.v[j], e);
#pragma unroll
                            for (int s = 0; s < EPV; ++s) {
                                const int idx = j * EPV + s - ch.h;
                                const uint32_t k = E::key(e[s]);
                                if (idx >= 0 && idx < ch.n && (k >> (shift + 8)) == pre)
                                    atomicAdd(&myh[(k >> shift) & 255u], 1u);
                            }
                        }
                        __syncthreads();
                        cur ^= 1;
                        if (tid < 256) {
                            uint32_t a = 0;
#pragma unroll
                            for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
                            chist[cur * 256 + tid] = a;
                        }
                        __syncthreads();
                        cluster.sync();
                        merge_plain(cluster, chist + cur * 256, S, g);
                        dt_find_bin<true>(g, need, &misc->bs);
                        const uint32_t dg = (uint32_t)misc->bs.digit;
                        need = misc->bs.need;
                        T_key |= dg << shift;
                        last_bin = (int)dg;
                        if (tid < S) misc->ceq[tid] = (int)cluster.map_shared_rank(chist, tid)[cur * 256 + dg];
                        __syncthreads();
                    }
                }
            } else {
                // the window holds fewer than Kc keys: full radix over the whole key
                need = Kc;
                T_key = 0;
                for (int rd = 0; rd < E::KB / 8; ++rd) {
                    const int shift = E::KB - 8 - 8 * rd;
                    const uint32_t pre = rd ? (T_key >> (shift + 8)) : 0u;
                    __syncthreads();
                    for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
                    __syncthreads();
                    for (int j = v0 + lane; j < v1; j += 32) {
                        T e[EPV];
                        ch.unpack(ch.v[j], e);
#pragma unroll
                        for (int s = 0; s < EPV; ++s) {
                            const int idx = j * EPV + s - ch.h;
                            const uint32_t k = E::key(e[s]);
                            if (idx >= 0 && idx < ch.n && (rd == 0 || (k >> (shift + 8)) == pre))
                                atomicAdd(&myh[(k >> shift) & 255u], 1u);
                        }
                    }
                    __syncthreads();
                    cur ^= 1;
                    if (tid < 256) {
                        uint32_t a = 0;
#pragma unroll
                        for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
                        chist[cur * 256 + tid] = a;
                    }
                    __syncthreads();
                    cluster.sync();
                    merge_plain(cluster, chist + cur * 256, S, g);
                    dt_find_bin<true>(g, need, &misc->bs);
                    const uint32_t dg = (uint32_t)misc->bs.digit;
                    need = misc->bs.need;
                    T_key |= dg << shift;
                    last_bin = (int)dg;
                    if (tid < S) misc->ceq[tid] = (int)cluster.map_shared_rank(chist, tid)[cur * 256 + dg];
                    __syncthreads();
                }
            }
            // threshold ties per warp slice, straight from the last round's histograms
            if (tid < NW) misc->weq[tid] = (last_bin >= 0 && last_bin < 256) ? (int)whist[tid * 256 + last_bin] : 0;
            __syncthreads();

            // emit keys above T, plus the first `need` ties by token id, into sel
            unsigned long long* sel = cand;
            int eqbase = 0;
            for (int j = 0; j < c; ++j) eqbase += misc->ceq[j];
            for (int w = 0; w < wid; ++w) eqbase += misc->weq[w];
            const float Tv = E::key_val(T_key);
            int running = 0;
            for (int base = v0; base < v1; base += 32) {
                const int j = base + lane;
                float x[EPV];
                int neq = 0;
                bool ok[EPV];
                if (j < v1) {
                    dt_vec_vals<T>(ch.v[j], x);
                    const bool full = (j >= full_lo && j < full_hi);
#pragma unroll
                    for (int s = 0; s < EPV; ++s) {
                        const int idx = j * EPV + s - ch.h;
                        ok[s] = full || (idx >= 0 && idx < ch.n);
                        neq += (ok[s] && x[s] == Tv);
                    }
                }
                const int inc = dt_warp_incl_scan(neq);
                int r = running + inc - neq;  // ties before this lane's vector in this warp slice
                running += __shfl_sync(0xffffffffu, inc, 31);
                if (j < v1) {
#pragma unroll
                    for (int s = 0; s < EPV; ++s) {
                        if (!ok[s] || !(x[s] >= Tv)) continue;
                        bool take = true;
                        if (x[s] == Tv) {
                            take = (eqbase + r < need);
                            ++r;
                        }
                        if (take) {
                            const int idx = j * EPV + s - ch.h;
                            const int slot = atomicAdd(&mp->nsel, 1);
                            if (slot < Kc)
                                sel[slot] = ((unsigned long long)E::key(dt_to_elem<T>(x[s])) << 32) |
                                            (unsigned long long)(0xFFFFFFFFu - (uint32_t)(lo + idx));
                        }
                    }
                }
            }
            __syncthreads();
            cluster.sync();
            // gather every CTA's selection (one warp per partner); this
            // overwrites the per-warp histograms, whose last read was before
            // the barrier
            if (tid < S) misc->cnsel[tid] = min(Kc, cluster.map_shared_rank(misc, tid)->pub[par].nsel);
            __syncthreads();
            for (int j = wid; j < S; j += NW) {
                int off = 0;
                for (int q = 0; q < j; ++q) off += misc->cnsel[q];
                const unsigned long long* rs = cluster.map_shared_rank(sel, j);
                const int cnt = misc->cnsel[j];
                for (int i = lane; i < cnt; i += 32)
                    if (off + i < Kc) all[off + i] = rs[i];
            }
            int tot = 0;
            for (int q = 0; q < S; ++q) tot += misc->cnsel[q];
            tot = min(tot, Kc);
            __syncthreads();
            if (tot > DT_SORT_MIN) dt_sort_and_write<T, NT>(all, tot, Kc, c, S, lse, row, cand_id, cand_lp);
            else dt_rank_and_write<T, NT>(sel, misc->cnsel[c], all, tot, Kc, lse, row, cand_id, cand_lp);
        }
        if (c == 0 && tid == 0) {
            int to = 0;
            for (int j = 0; j < S; ++j) to |= misc->pin[j].timeout;
            lse_out[row] = to ? __int_as_float(0x7FC00000) : lse;
        }
        // the next row's copy starts once every read of this one is done
        if (nxt < rows) {
            __syncthreads();
            dt_fence_proxy_async();
            issue(nxt);
        }
    }
    // after a fallback, partners may still be gathering from this CTA's
    // shared memory (every CTA took the same rows down the same branches)
    if (fallback_taken) {
        __syncthreads();
        cluster.sync();
    }
}

}  // namespace

cudaError_t dt_kn1_set_probe(long long budget) {
    return cudaMemcpyToSymbol(g_kn1_probe, &budget, sizeof(budget));
}

size_t dt_kn1_smem_bytes(int chunk, int Kc, int esize) {
    (void)Kc;  // the fixed candidate buffers also hold the fallback's Kc <= 1024 selections
    return OFF_DATA + (size_t)chunk * esize + 32;
}

// Sets the kernel's shared-memory and cluster-size attributes for a launch.
template <typename T>
cudaError_t kn1_prepare(int S, size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(kn1_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && S > 8) e = cudaFuncSetAttribute(kn1_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

int dt_kn1_max_clusters(int dtype, int S, int chunk, int Kc) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const size_t smem = dt_kn1_smem_bytes(chunk, Kc, esize);
    if (dtype == DT_BF16) {
        if (kn1_prepare<uint16_t>(S, smem) != cudaSuccess) return 0;
        return dt_max_active_clusters(kn1_kernel<uint16_t>, S, NT, smem);
    }
    if (kn1_prepare<float>(S, smem) != cudaSuccess) return 0;
    return dt_max_active_clusters(kn1_kernel<float>, S, NT, smem);
}

cudaError_t dt_kn1_launch(const void* logits, int dtype, int rows, int grid_rows, int V, int Kc, int S, int chunk,
                          float* lse, int32_t* cand_id, float* cand_lp, cudaStream_t st) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const size_t smem = dt_kn1_smem_bytes(chunk, Kc, esize);
    DtLaunch lc(dim3(S, grid_rows, 1), dim3(NT, 1, 1), smem, st, S);
    cudaError_t e;
    if (dtype == DT_BF16) {
        if ((e = kn1_prepare<uint16_t>(S, smem)) != cudaSuccess) return e;
        return cudaLaunchKernelEx(&lc.cfg, kn1_kernel<uint16_t>, (const uint16_t*)logits, V, chunk, Kc, rows,
                                  lse, cand_id, cand_lp);
    }
    if ((e = kn1_prepare<float>(S, smem)) != cudaSuccess) return e;
    return cudaLaunchKernelEx(&lc.cfg, kn1_kernel<float>, (const float*)logits, V, chunk, Kc, rows, lse,
                              cand_id, cand_lp);
}
