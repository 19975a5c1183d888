// kn1_candidates.cu -- stage 1: per-position log-softmax and exact Top-Kc.
//
// [DARTree] Algorithm 1, its per-position Top-K candidate step; [DDTree] section 3.3
// (log-domain scores of each position's Top-K tokens).
//
// One thread-block cluster of S CTAs per row (request b, position l); CTA c
// owns a contiguous vocabulary chunk.  Each CTA streams its chunk once from
// HBM into shared memory with a 1-D bulk async copy, then, reading shared
// memory 16 bytes per lane at a time:
//   pass 1  chunk max (order key);
//   pass 2  sum exp(x - max) and a 256-bin histogram of the keys within 256
//           key steps below the chunk max (one histogram per warp, warp w
//           owning a contiguous slice of the chunk);
//   cluster exchange (DSMEM) -> row log-normaliser and the exact Kc-th key;
//   (fp32 logits: two more 8-bit radix rounds on the low key bits; rows where
//    the 256-step window holds fewer than Kc keys: full radix from the top);
//   emit the CTA's keys above the threshold, plus threshold ties taken in
//   token-id order (per-warp tie counts come from the histograms, the order
//   inside a warp from a warp scan);
//   gather the Kc selected (key, id) pairs of all CTAs (one warp per partner)
//   and write each own entry at its rank (one warp per entry).
// Every element of the row is read from HBM exactly once; nothing goes to
// global memory except the outputs.  A row whose staging wait ran out of its
// bound gets a NaN normaliser (the selection kernels turn that into
// DT_DEV_TIMEOUT).
#include <cuda_bf16.h>

#include "dt_device.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int SMAX = 16;

struct Kn1Misc {
    uint64_t bar;
    float m;           // chunk max value
    float s;           // chunk sum exp(x - m)
    uint32_t mk16;     // chunk max key, top 16 bits
    int nsel;          // selected entries in this CTA
    int timeout;
    float cm[SMAX];    // partners' values, copied through DSMEM
    float cs[SMAX];
    uint32_t cmk[SMAX];
    int ceq[SMAX];
    int cnsel[SMAX];
    int cto[SMAX];
    float lse;
    int round_digit;
    int round_need;
    int weq[NW];       // threshold ties per warp slice
    float red_f[NW];   // per-warp maxima
    float red_s[NW];   // per-warp sums
    int wsum[8];
};

// Dynamic shared memory: [misc 1 KB][per-warp histograms NW*1 KB][chist 2 KB]
// [sel Kc*8][all Kc*8][chunk data + 16]
DT_DI uint32_t* whist_of(unsigned char* s) { return (uint32_t*)(s + 1024); }
DT_DI uint32_t* chist_of(unsigned char* s) { return (uint32_t*)(s + 1024 + NW * 1024); }
DT_DI unsigned long long* sel_of(unsigned char* s) { return (unsigned long long*)(s + 1024 + NW * 1024 + 2048); }

// Vector access to the staged chunk: vector j (16 bytes) holds elements
// j*EPV - h .. j*EPV - h + EPV - 1, where h is the head misalignment.
template <typename T>
struct Chunk {
    static constexpr int EPV = 16 / sizeof(T);
    const uint4* v;  // 16-byte aligned base
    int h;           // elements of vector 0 that precede the chunk
    int n;           // elements in the chunk
    int nv;          // vectors covering the chunk
    int lo;          // token id of element 0
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

// Hardware base-2 exponential (approximate, ~2 ulp), used only for the
// fp32 normaliser sum whose tolerance is 1e-5.
DT_DI float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The element type's bits of a value that came from that type (exact).
template <typename T> DT_DI T to_elem(float x);
template <> DT_DI uint16_t to_elem<uint16_t>(float x) { return (uint16_t)(__float_as_uint(x) >> 16); }
template <> DT_DI float to_elem<float>(float x) { return x; }

// Values of the EPV elements of a 16-byte vector, as fp32.
template <typename T> DT_DI void vec_vals(const uint4& q, float (&x)[16 / sizeof(T)]);
template <> DT_DI void vec_vals<uint16_t>(const uint4& q, float (&x)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}
template <> DT_DI void vec_vals<float>(const uint4& q, float (&x)[4]) {
    x[0] = __uint_as_float(q.x);
    x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z);
    x[3] = __uint_as_float(q.w);
}

// Largest value in a full 16-byte vector (bf16: packed two-way compares).
template <typename T> DT_DI float vec_max(const uint4& q);
template <> DT_DI float vec_max<uint16_t>(const uint4& q) {
    const __nv_bfloat162 a = __hmax2(*(const __nv_bfloat162*)&q.x, *(const __nv_bfloat162*)&q.y);
    const __nv_bfloat162 b = __hmax2(*(const __nv_bfloat162*)&q.z, *(const __nv_bfloat162*)&q.w);
    const __nv_bfloat162 c = __hmax2(a, b);
    return fmaxf(__low2float(c), __high2float(c));
}
template <> DT_DI float vec_max<float>(const uint4& q) {
    return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)), fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
}

// Warp w owns vectors [w*vseg, min(nv, (w+1)*vseg)).
DT_DI void warp_vectors(int nv, int* v0, int* v1) {
    const int w = threadIdx.x >> 5;
    const int vseg = (nv + NW - 1) / NW;
    *v0 = min(nv, w * vseg);
    *v1 = min(nv, *v0 + vseg);
}

// Block-wide: global histogram g[256]; when TOP_IS_HIGH a higher bin index is
// a larger key, else bin 0 is the largest.  Finds the bin holding the
// need-th largest key: misc->round_digit (-1 if the bins hold fewer than
// `need` keys) and misc->round_need (keys still needed inside that bin).
template <bool TOP_IS_HIGH>
DT_DI void find_bin(const uint32_t* g, int need, Kn1Misc* misc) {
    const int t = threadIdx.x;
    int v = 0;
    if (t < 256) v = (int)g[TOP_IS_HIGH ? 255 - t : t];
    const int inc = dt_warp_incl_scan(v);
    if (t < 256 && (t & 31) == 31) misc->wsum[t >> 5] = inc;
    if (t == 0) { misc->round_digit = -1; misc->round_need = need; }
    __syncthreads();
    if (t < 256) {
        int before = 0;
        for (int i = 0; i < (t >> 5); ++i) before += misc->wsum[i];
        const int cum = before + inc;
        if (cum >= need && cum - v < need) {
            misc->round_digit = TOP_IS_HIGH ? 255 - t : t;
            misc->round_need = need - (cum - v);
        }
    }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(NT) kn1_kernel(const T* __restrict__ logits, int V, int chunk, int Kc,
                                                 int L, float* __restrict__ lse_out,
                                                 int32_t* __restrict__ cand_id,
                                                 float* __restrict__ cand_lp) {
    using E = DtElem<T>;
    constexpr int EPV = Chunk<T>::EPV;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t g[256];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int c = (int)cluster.block_rank();
    const int row = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int lo = min(V, c * chunk), hi = min(V, lo + chunk);

    Kn1Misc* misc = (Kn1Misc*)smem;
    uint32_t* whist = whist_of(smem);
    uint32_t* chist = chist_of(smem);
    unsigned long long* sel = sel_of(smem);
    unsigned long long* all = sel + Kc;
    unsigned char* dbase = (unsigned char*)(all + Kc);

    if (tid == 0) {
        dt_mbar_init(&misc->bar, 1);
        dt_fence_mbar_init();
        misc->nsel = 0;
        misc->timeout = 0;
    }
    for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
    dt_pdl_trigger();
    __syncthreads();
    dt_pdl_wait();  // the logits may come from the kernel just before us

    // ---- stage the chunk (one HBM read) --------------------------------
    uint32_t bulk = 0;
    const T* rowp = logits + (size_t)row * (size_t)V;
    const T* xs = dt_stage_row<T>(rowp, lo, hi, dbase, &misc->bar, &bulk);
    // one thread waits on the copy; the others block in the barrier below
    // (blocked warps take no issue slots)
    if (bulk && tid == 0) {
        if (!dt_mbar_wait(&misc->bar, 0)) {
            misc->timeout = 1;
            dt_mbar_wait(&misc->bar, 0);
        }
    }
    __syncthreads();
    Chunk<T> ch;
    ch.h = (int)(((uintptr_t)xs - (uintptr_t)dbase) / sizeof(T));
    ch.v = (const uint4*)dbase;
    ch.n = hi - lo;
    ch.nv = (ch.h + ch.n + EPV - 1) / EPV;
    ch.lo = lo;
    int v0, v1;
    warp_vectors(ch.nv, &v0, &v1);

    // ---- pass 1: chunk max (packed compares on whole vectors) -------------
    // vectors 0 and nv-1 may be partial (misaligned head, ragged tail); they
    // take the element-wise path
    const int full_lo = (ch.h > 0) ? 1 : 0;
    const int full_hi = ((ch.h + ch.n) % EPV == 0) ? ch.nv : ch.nv - 1;
    float mx = -__int_as_float(0x7F800000);
    for (int j = v0 + lane; j < v1; j += 32) {
        const uint4 q = ch.v[j];
        if (j >= full_lo && j < full_hi) {
            mx = fmaxf(mx, vec_max<T>(q));
        } else {
            T e[EPV];
            ch.unpack(q, e);
#pragma unroll
            for (int s = 0; s < EPV; ++s) {
                const int idx = j * EPV + s - ch.h;
                if (idx >= 0 && idx < ch.n) mx = fmaxf(mx, E::val(e[s]));
            }
        }
    }
    mx = dt_warp_max(mx);
    if (lane == 0) misc->red_f[wid] = mx;
    __syncthreads();
    float m_c = -__int_as_float(0x7F800000);
#pragma unroll
    for (int w = 0; w < NW; ++w) m_c = fmaxf(m_c, misc->red_f[w]);
    const bool any = ch.n > 0;
    const uint32_t mk16 = any ? (E::key(to_elem<T>(m_c)) >> (E::KB - 16)) : 0u;
    const bool finite_max = (m_c != -__int_as_float(0x7F800000));
    // the window holds keys mk16-255 .. mk16 (top 16 bits); as a value bound
    const uint32_t klo = mk16 >= 255u ? mk16 - 255u : 0u;
    const float x_lo = (klo <= 127u) ? -__int_as_float(0x7F800000) : E::key_val(klo << (E::KB - 16));

    // ---- pass 2: sum exp(x - max) and the windowed key histogram ---------
    const float log2e = 1.44269504088896340736f;
    float sum = 0.f;
    uint32_t* myh = whist + wid * 256;
    for (int j = v0 + lane; j < v1; j += 32) {
        const uint4 q = ch.v[j];
        float x[EPV];
        vec_vals<T>(q, x);
        const bool full = (j >= full_lo && j < full_hi);
#pragma unroll
        for (int s = 0; s < EPV; ++s) {
            const int idx = j * EPV + s - ch.h;
            if (full || (idx >= 0 && idx < ch.n)) {
                // x - max is exact for the max itself (e^0 = 1 at any magnitude)
                if (finite_max) sum += ex2_approx(__fmul_rn(__fsub_rn(x[s], m_c), log2e));
                if (x[s] >= x_lo) atomicAdd(&myh[mk16 - (E::key(to_elem<T>(x[s])) >> (E::KB - 16))], 1u);
            }
        }
    }
    sum = dt_warp_sum(sum);
    if (lane == 0) misc->red_s[wid] = sum;
    __syncthreads();
    if (tid < 256) {
        uint32_t a = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
        chist[tid] = a;
    }
    if (tid == 0) {
        float a = 0.f;
        for (int i = 0; i < NW; ++i) a += misc->red_s[i];
        misc->s = a;
        misc->m = m_c;
        misc->mk16 = mk16;
    }
    __syncthreads();
    cluster.sync();

    // ---- exchange: normaliser and window histogram ------------------------
    if (tid < S) {
        const Kn1Misc* r = cluster.map_shared_rank(misc, tid);
        misc->cm[tid] = r->m;
        misc->cs[tid] = r->s;
        misc->cmk[tid] = r->mk16;
        misc->cto[tid] = r->timeout;
    }
    __syncthreads();
    uint32_t Mk16 = 0;
    for (int j = 0; j < S; ++j) Mk16 = max(Mk16, misc->cmk[j]);
    if (tid == 0) {
        float M = misc->cm[0];
        for (int j = 1; j < S; ++j) M = fmaxf(M, misc->cm[j]);
        float ssum = 0.f;
        for (int j = 0; j < S; ++j)
            if (misc->cm[j] != -__int_as_float(0x7F800000)) ssum += misc->cs[j] * __expf(misc->cm[j] - M);
        misc->lse = M + logf(ssum);
    }
    // global window histogram: bin t counts keys whose top 16 bits equal Mk16 - t
    if (tid < 256) {
        uint32_t part[SMAX];
#pragma unroll
        for (int j = 0; j < SMAX; ++j) {
            part[j] = 0;
            const int wj = tid - (int)(Mk16 - misc->cmk[j < S ? j : 0]);
            if (j < S && wj >= 0 && wj < 256) part[j] = cluster.map_shared_rank(chist, j)[wj];
        }
        uint32_t a = 0;
#pragma unroll
        for (int j = 0; j < SMAX; ++j) a += part[j];
        g[tid] = a;
    }
    __syncthreads();
    find_bin<false>(g, Kc, misc);

    uint32_t T_key;
    int need;
    int cur = 0;        // chist buffer of the last round
    int last_bin = -1;  // per-warp histogram bin holding the threshold ties
    if (misc->round_digit >= 0) {
        const uint32_t t16 = Mk16 - (uint32_t)misc->round_digit;
        need = misc->round_need;
        if (tid < S) {
            const int wj = (int)(misc->cmk[tid] - t16);
            misc->ceq[tid] = (wj >= 0 && wj < 256) ? (int)cluster.map_shared_rank(chist, tid)[wj] : 0;
        }
        last_bin = (int)(mk16 - t16);  // may be outside [0,256) when this CTA has no ties
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
                if (tid < 256) {
                    uint32_t part[SMAX];
#pragma unroll
                    for (int j = 0; j < SMAX; ++j)
                        part[j] = (j < S) ? cluster.map_shared_rank(chist, j)[cur * 256 + tid] : 0u;
                    uint32_t a = 0;
#pragma unroll
                    for (int j = 0; j < SMAX; ++j) a += part[j];
                    g[tid] = a;
                }
                __syncthreads();
                find_bin<true>(g, need, misc);
                const uint32_t dg = (uint32_t)misc->round_digit;
                need = misc->round_need;
                T_key |= dg << shift;
                last_bin = (int)dg;
                if (tid < S) misc->ceq[tid] = (int)cluster.map_shared_rank(chist, tid)[cur * 256 + dg];
                __syncthreads();
            }
        }
    } else {
        // fallback: full radix select over the whole key, 8 bits per round
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
            if (tid < 256) {
                uint32_t part[SMAX];
#pragma unroll
                for (int j = 0; j < SMAX; ++j)
                    part[j] = (j < S) ? cluster.map_shared_rank(chist, j)[cur * 256 + tid] : 0u;
                uint32_t a = 0;
#pragma unroll
                for (int j = 0; j < SMAX; ++j) a += part[j];
                g[tid] = a;
            }
            __syncthreads();
            find_bin<true>(g, need, misc);
            const uint32_t dg = (uint32_t)misc->round_digit;
            need = misc->round_need;
            T_key |= dg << shift;
            last_bin = (int)dg;
            if (tid < S) misc->ceq[tid] = (int)cluster.map_shared_rank(chist, tid)[cur * 256 + dg];
            __syncthreads();
        }
    }
    // threshold ties per warp slice, straight from the last round's histograms
    if (tid < NW) misc->weq[tid] = (last_bin >= 0 && last_bin < 256) ? (int)whist[tid * 256 + last_bin] : 0;
    __syncthreads();

    // ---- emit: keys above T, plus the first `need` ties by token id -------
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
            vec_vals<T>(ch.v[j], x);
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
                    const int slot = atomicAdd(&misc->nsel, 1);
                    if (slot < Kc)
                        sel[slot] = ((unsigned long long)E::key(to_elem<T>(x[s])) << 32) |
                                    (unsigned long long)(0xFFFFFFFFu - (uint32_t)(lo + idx));
                }
            }
        }
    }
    __syncthreads();
    cluster.sync();

    // ---- gather every CTA's selection (one warp per partner) -------------
    if (tid < S) misc->cnsel[tid] = min(Kc, cluster.map_shared_rank(misc, tid)->nsel);
    __syncthreads();
    for (int j = wid; j < S; j += NW) {
        int off = 0;
        for (int q = 0; q < j; ++q) off += misc->cnsel[q];
        const unsigned long long* rs = cluster.map_shared_rank(sel, j);
        const int cnt = misc->cnsel[j];
        for (int i = lane; i < cnt; i += 32)
            if (off + i < Kc) all[off + i] = rs[i];
    }
    int total = 0;
    for (int q = 0; q < S; ++q) total += misc->cnsel[q];
    total = min(total, Kc);
    __syncthreads();
    cluster.sync();  // partners' selections are no longer read after this point

    // ---- rank each own entry (one warp per entry) and write it -----------
    const float lse = misc->lse;
    const int mine = misc->cnsel[c];
    for (int i = wid; i < mine; i += NW) {
        const unsigned long long key = sel[i];
        int rank = 0;
        for (int q = lane; q < total; q += 32) rank += (all[q] > key);
        rank = dt_warp_sum_i(rank);
        if (lane == 0 && rank < Kc) {
            const uint32_t id = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
            const float v = E::key_val((uint32_t)(key >> 32));
            cand_id[(size_t)row * Kc + rank] = (int32_t)id;
            cand_lp[(size_t)row * Kc + rank] = __fsub_rn(v, lse);
        }
    }
    if (c == 0 && tid == 0) {
        int to = 0;
        for (int j = 0; j < S; ++j) to |= misc->cto[j];
        lse_out[row] = to ? __int_as_float(0x7FC00000) : lse;
    }
}

}  // namespace

size_t dt_kn1_smem_bytes(int chunk, int Kc, int esize) {
    return 1024 + (size_t)NW * 1024 + 2048 + (size_t)Kc * 16 + (size_t)chunk * esize + 32;
}

cudaError_t dt_kn1_launch(const void* logits, int dtype, int rows, int L, int V, int Kc, int S, int chunk,
                          float* lse, int32_t* cand_id, float* cand_lp, cudaStream_t st) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const size_t smem = dt_kn1_smem_bytes(chunk, Kc, esize);
    DtLaunch lc(dim3(S, rows, 1), dim3(NT, 1, 1), smem, st, S);
    cudaError_t e;
    if (dtype == DT_BF16) {
        auto k = kn1_kernel<uint16_t>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        if (S > 8 && (e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        return cudaLaunchKernelEx(&lc.cfg, k, (const uint16_t*)logits, V, chunk, Kc, L, lse, cand_id, cand_lp);
    } else {
        auto k = kn1_kernel<float>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        if (S > 8 && (e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        return cudaLaunchKernelEx(&lc.cfg, k, (const float*)logits, V, chunk, Kc, L, lse, cand_id, cand_lp);
    }
}
