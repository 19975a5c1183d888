// kn1_candidates.cu -- stage 1: per-position log-softmax and exact Top-Kc.
//
// [DARTree] Algorithm 1 line 4 (C_d = TopK(L_d^base, K)); [DDTree] section 3.3
// (log-domain scores of each position's Top-K tokens).
//
// One thread-block cluster of S CTAs per row (request b, position l); CTA c
// owns a contiguous vocabulary chunk.  Each CTA streams its chunk once from
// HBM into shared memory with a 1-D bulk async copy, then:
//   pass 1  chunk max (value and order key);
//   pass 2  sum exp(x - max) and a 256-bin histogram of the keys within 256
//           key steps below the chunk max (per-warp privatised);
//   cluster exchange (DSMEM) -> row log-normaliser and the exact Kc-th key;
//   (fp32 logits: two more 8-bit radix rounds on the low key bits; rows where
//    the 256-step window holds fewer than Kc keys: full radix from the top);
//   emit the CTA's keys above the threshold, plus threshold ties taken by
//   ascending token id (stable warp ballots across the cluster);
//   gather the Kc selected (key, id) pairs from every CTA and write each at
//   its rank (logit descending, token id ascending).
// Every element of the row is read from HBM exactly once; nothing goes to
// global memory except the outputs.
#include "dt_device.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT = 256;
constexpr int NW = NT / 32;

struct Kn1Misc {
    uint64_t bar;
    float m;           // chunk max value
    float s;           // chunk sum exp(x - m)
    uint32_t mk16;     // chunk max key, top 16 bits
    int nsel;          // selected entries in this CTA
    int timeout;
    // per-cluster copies read through DSMEM
    float cm[16];
    float cs[16];
    uint32_t cmk[16];
    int ceq[16];
    int cnsel[16];
    // results of the threshold search (identical in every CTA)
    float lse;
    uint32_t T;        // full threshold key
    int need;          // threshold ties to take (smallest ids first)
    int eq_before;     // threshold ties in lower-ranked CTAs
    int round_digit;
    int round_need;
    int window_ok;
    int red_i[NW];
    float red_f[NW];
    uint32_t red_u[NW];
};

template <typename T>
struct Kn1Smem {
    // layout in dynamic shared memory
    static DT_DI Kn1Misc* misc(unsigned char* s) { return (Kn1Misc*)s; }
    static DT_DI uint32_t* whist(unsigned char* s) { return (uint32_t*)(s + 1024); }           // [NW][256]
    static DT_DI uint32_t* chist(unsigned char* s) { return (uint32_t*)(s + 1024 + NW * 1024); } // [2][256]
    static DT_DI unsigned long long* sel(unsigned char* s) {
        return (unsigned long long*)(s + 1024 + NW * 1024 + 2048);
    }
    static DT_DI unsigned long long* all(unsigned char* s, int Kc) { return sel(s) + Kc; }
    static DT_DI unsigned char* data(unsigned char* s, int Kc) {
        return (unsigned char*)(all(s, Kc) + Kc);
    }
};

// Warp w owns elements [w*seg, min(n, (w+1)*seg)) of the chunk.
DT_DI void warp_segment(int n, int* s0, int* s1) {
    const int w = threadIdx.x >> 5;
    const int seg = (n + NW - 1) / NW;
    *s0 = min(n, w * seg);
    *s1 = min(n, *s0 + seg);
}

// Block-wide: given a global histogram g[256] (bins ordered so that a HIGHER
// bin index is a LARGER key when `top_is_high`, else bin 0 is the largest),
// find the bin holding the need-th largest key.  Returns via misc
// round_digit / round_need (count still needed inside that bin).
template <bool TOP_IS_HIGH>
DT_DI void find_bin(const uint32_t* g, int need, Kn1Misc* misc) {
    // thread t < 256 holds bin b(t) ordered from the largest key downwards
    __shared__ int wsum[8];
    const int t = threadIdx.x;
    int v = 0;
    if (t < 256) v = (int)g[TOP_IS_HIGH ? 255 - t : t];
    int inc = dt_warp_incl_scan(v);
    if (t < 256 && (t & 31) == 31) wsum[t >> 5] = inc;
    __syncthreads();
    int before = 0;
    if (t < 256)
        for (int i = 0; i < (t >> 5); ++i) before += wsum[i];
    int cum = before + inc;  // count of keys in bins up to and including t (from the top)
    if (t == 0) { misc->round_digit = -1; misc->round_need = need; }
    __syncthreads();
    if (t < 256 && cum >= need && cum - v < need) {
        misc->round_digit = TOP_IS_HIGH ? 255 - t : t;
        misc->round_need = need - (cum - v);
    }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(NT) kn1_kernel(const T* __restrict__ logits, int V, int chunk, int Kc,
                                                 int L, float* __restrict__ lse_out,
                                                 int32_t* __restrict__ cand_id,
                                                 float* __restrict__ cand_lp, int32_t* __restrict__ status) {
    using E = DtElem<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int c = (int)cluster.block_rank();
    const int row = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int lo = min(V, c * chunk), hi = min(V, lo + chunk);
    const int n = hi - lo;

    Kn1Misc* misc = Kn1Smem<T>::misc(smem);
    uint32_t* whist = Kn1Smem<T>::whist(smem);
    uint32_t* chist = Kn1Smem<T>::chist(smem);
    unsigned long long* sel = Kn1Smem<T>::sel(smem);
    unsigned long long* all = Kn1Smem<T>::all(smem, Kc);
    unsigned char* dbase = Kn1Smem<T>::data(smem, Kc);

    if (tid == 0) {
        dt_mbar_init(&misc->bar, 1);
        dt_fence_mbar_init();
        misc->nsel = 0;
        misc->timeout = 0;
    }
    for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
    __syncthreads();

    // ---- stage the chunk (one HBM read) --------------------------------
    uint32_t bulk = 0;
    const T* rowp = logits + (size_t)row * (size_t)V;
    const T* x = dt_stage_row<T>(rowp, lo, hi, dbase, &misc->bar, &bulk);
    if (bulk) {
        if (!dt_mbar_wait(&misc->bar, 0)) {
            misc->timeout = 1;  // benign race: every writer stores 1
            dt_mbar_wait(&misc->bar, 0);
        }
    }
    __syncthreads();

    int s0, s1;
    warp_segment(n, &s0, &s1);

    // ---- pass 1: chunk max ----------------------------------------------
    float mx = -__int_as_float(0x7F800000);
    uint32_t mk = 0;
    for (int e = s0 + lane; e < s1; e += 32) {
        T v = x[e];
        mx = fmaxf(mx, E::val(v));
        mk = max(mk, E::key(v));
    }
    mx = dt_warp_max(mx);
    mk = dt_warp_max_u32(mk);
    if (lane == 0) { misc->red_f[wid] = mx; misc->red_u[wid] = mk; }
    __syncthreads();
    if (tid == 0) {
        float a = misc->red_f[0];
        uint32_t b = misc->red_u[0];
        for (int i = 1; i < NW; ++i) { a = fmaxf(a, misc->red_f[i]); b = max(b, misc->red_u[i]); }
        misc->m = a;
        misc->mk16 = (n > 0) ? (b >> (E::KB - 16)) : 0u;
    }
    __syncthreads();
    const float m_c = misc->m;
    const uint32_t mk16 = misc->mk16;
    const bool finite_max = (m_c != -__int_as_float(0x7F800000));

    // ---- pass 2: sum exp and the windowed key histogram -----------------
    float sum = 0.f;
    uint32_t* myh = whist + wid * 256;
    for (int e = s0 + lane; e < s1; e += 32) {
        T v = x[e];
        if (finite_max) sum += __expf(E::val(v) - m_c);
        uint32_t k16 = E::key(v) >> (E::KB - 16);
        uint32_t w = mk16 - k16;
        if (w < 256u) atomicAdd(&myh[w], 1u);
    }
    sum = dt_warp_sum(sum);
    if (lane == 0) misc->red_f[wid] = sum;
    __syncthreads();
    if (tid < 256) {
        uint32_t a = 0;
        for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
        chist[tid] = a;  // buffer 0
    }
    if (tid == 0) {
        float a = 0.f;
        for (int i = 0; i < NW; ++i) a += misc->red_f[i];
        misc->s = a;
    }
    __syncthreads();
    cluster.sync();

    // ---- exchange: normaliser and window histogram ------------------------
    if (tid < S) {
        Kn1Misc* r = cluster.map_shared_rank(misc, tid);
        misc->cm[tid] = r->m;
        misc->cs[tid] = r->s;
        misc->cmk[tid] = r->mk16;
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
    // global window histogram: bin t counts keys equal to Mk16 - t
    uint32_t* g = whist;  // per-warp histograms are summed already; reuse the space
    __syncthreads();
    if (tid < 256) {
        uint32_t a = 0;
        for (int j = 0; j < S; ++j) {
            int wj = tid - (int)(Mk16 - misc->cmk[j]);
            if (wj >= 0 && wj < 256) {
                const uint32_t* rh = cluster.map_shared_rank(chist, j);
                a += rh[wj];
            }
        }
        g[tid] = a;
    }
    __syncthreads();
    find_bin<false>(g, Kc, misc);

    uint32_t T_key;
    int need;
    int cur = 0;  // histogram buffer parity of the last round
    if (misc->round_digit >= 0) {
        // threshold's top 16 key bits found in the window
        const uint32_t t16 = Mk16 - (uint32_t)misc->round_digit;
        need = misc->round_need;
        // ties at t16 per CTA (for bf16 these are the final ties)
        if (tid < S) {
            int wj = (int)(misc->cmk[tid] - t16);
            int e = 0;
            if (wj >= 0 && wj < 256) {
                const uint32_t* rh = cluster.map_shared_rank(chist, tid);
                e = (int)rh[wj];
            }
            misc->ceq[tid] = e;
        }
        T_key = t16 << (E::KB - 16);
        if (E::KB == 32) {
            // two radix rounds over the low 16 bits among keys with top bits t16
            for (int rd = 0; rd < 2; ++rd) {
                const int shift = 8 - 8 * rd;  // digit bits [shift, shift+8)
                const uint32_t pre = T_key >> (shift + 8);
                __syncthreads();
                for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
                __syncthreads();
                for (int e = s0 + lane; e < s1; e += 32) {
                    uint32_t k = E::key(x[e]);
                    if ((k >> (shift + 8)) == pre) atomicAdd(&whist[wid * 256 + ((k >> shift) & 255u)], 1u);
                }
                __syncthreads();
                cur ^= 1;
                if (tid < 256) {
                    uint32_t a = 0;
                    for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
                    chist[cur * 256 + tid] = a;
                }
                __syncthreads();
                cluster.sync();
                __shared__ uint32_t gg[256];
                if (tid < 256) {
                    uint32_t a = 0;
                    for (int j = 0; j < S; ++j) a += cluster.map_shared_rank(chist, j)[cur * 256 + tid];
                    gg[tid] = a;
                }
                __syncthreads();
                find_bin<true>(gg, need, misc);
                const uint32_t dg = (uint32_t)misc->round_digit;
                need = misc->round_need;
                T_key |= dg << shift;
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
            const int pbits = 8 * rd;
            const uint32_t pre = pbits ? (T_key >> (shift + 8)) : 0u;
            __syncthreads();
            for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
            __syncthreads();
            for (int e = s0 + lane; e < s1; e += 32) {
                uint32_t k = E::key(x[e]);
                if (pbits == 0 || (k >> (shift + 8)) == pre)
                    atomicAdd(&whist[wid * 256 + ((k >> shift) & 255u)], 1u);
            }
            __syncthreads();
            cur ^= 1;
            if (tid < 256) {
                uint32_t a = 0;
                for (int w = 0; w < NW; ++w) a += whist[w * 256 + tid];
                chist[cur * 256 + tid] = a;
            }
            __syncthreads();
            cluster.sync();
            __shared__ uint32_t gf[256];
            if (tid < 256) {
                uint32_t a = 0;
                for (int j = 0; j < S; ++j) a += cluster.map_shared_rank(chist, j)[cur * 256 + tid];
                gf[tid] = a;
            }
            __syncthreads();
            find_bin<true>(gf, need, misc);
            const uint32_t dg = (uint32_t)misc->round_digit;
            need = misc->round_need;
            T_key |= dg << shift;
            if (tid < S) misc->ceq[tid] = (int)cluster.map_shared_rank(chist, tid)[cur * 256 + dg];
            __syncthreads();
        }
    }
    __syncthreads();

    // ---- emit: keys above T, plus the first `need` ties by token id -------
    int eq_before = 0;
    for (int j = 0; j < c; ++j) eq_before += misc->ceq[j];
    // per-warp tie counts in this CTA (warp segments are in id order)
    int my_eq = 0;
    for (int e = s0 + lane; e < s1; e += 32) my_eq += (E::key(x[e]) == T_key);
    my_eq = dt_warp_sum_i(my_eq);
    if (lane == 0) misc->red_i[wid] = my_eq;
    __syncthreads();
    int eqbase = eq_before;
    for (int w = 0; w < wid; ++w) eqbase += misc->red_i[w];
    int running = 0;
    for (int base = s0; base < s1; base += 32) {
        const int e = base + lane;
        const bool valid = e < s1;
        const uint32_t k = valid ? E::key(x[e]) : 0u;
        const bool gt = valid && k > T_key;
        const bool eq = valid && k == T_key;
        const unsigned bal = __ballot_sync(0xffffffffu, eq);
        const int r = running + __popc(bal & ((1u << lane) - 1u));
        running += __popc(bal);
        if (gt || (eq && eqbase + r < need)) {
            int slot = atomicAdd(&misc->nsel, 1);
            if (slot < Kc)
                sel[slot] = ((unsigned long long)k << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)(lo + e));
        }
    }
    __syncthreads();
    cluster.sync();

    // ---- gather every CTA's selection and write each entry at its rank ---
    if (tid < S) misc->cnsel[tid] = min(Kc, cluster.map_shared_rank(misc, tid)->nsel);
    __syncthreads();
    int off = 0;
    for (int j = 0; j < S; ++j) {
        const int cnt = misc->cnsel[j];
        const unsigned long long* rs = cluster.map_shared_rank(sel, j);
        for (int i = tid; i < cnt; i += NT)
            if (off + i < Kc) all[off + i] = rs[i];
        off += cnt;
    }
    const int total = min(off, Kc);
    __syncthreads();
    cluster.sync();  // remote selections no longer needed after this point

    const float lse = misc->lse;
    const int mine = misc->cnsel[c];
    for (int i = tid; i < mine; i += NT) {
        const unsigned long long key = sel[i];
        int rank = 0;
        for (int j = 0; j < total; ++j) rank += (all[j] > key);
        const uint32_t id = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
        const float v = E::key_val((uint32_t)(key >> 32));
        if (rank < Kc) {
            cand_id[(size_t)row * Kc + rank] = (int32_t)id;
            cand_lp[(size_t)row * Kc + rank] = __fsub_rn(v, lse);
        }
    }
    if (c == 0 && tid == 0) {
        lse_out[row] = lse;
        if (misc->timeout) atomicOr(&status[row / L], DT_DEV_TIMEOUT);
    }
    if (c != 0 && tid == 0 && misc->timeout) atomicOr(&status[row / L], DT_DEV_TIMEOUT);
}

}  // namespace

size_t dt_kn1_smem_bytes(int chunk, int Kc, int esize) {
    return 1024 + (size_t)NW * 1024 + 2048 + (size_t)Kc * 16 + (size_t)chunk * esize + 16;
}

cudaError_t dt_kn1_launch(const void* logits, int dtype, int rows, int L, int V, int Kc, int S, int chunk,
                          float* lse, int32_t* cand_id, float* cand_lp, int32_t* status, cudaStream_t st) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    const size_t smem = dt_kn1_smem_bytes(chunk, Kc, esize);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, rows, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (dtype == DT_BF16) {
        auto k = kn1_kernel<uint16_t>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        if (S > 8 && (e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        return cudaLaunchKernelEx(&cfg, k, (const uint16_t*)logits, V, chunk, Kc, L, lse, cand_id, cand_lp, status);
    } else {
        auto k = kn1_kernel<float>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        if (S > 8 && (e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        return cudaLaunchKernelEx(&cfg, k, (const float*)logits, V, chunk, Kc, L, lse, cand_id, cand_lp, status);
    }
}
