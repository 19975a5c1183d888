// dt_device.cuh -- device helpers shared by the draft-tree kernels (sm_103a).
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dtree.h"

namespace cg = cooperative_groups;

#define DT_DI __device__ __forceinline__

// Bounded waits give up after this many SM clock cycles (~1 s at 2 GHz) and
// report DT_DEV_TIMEOUT instead of spinning forever.
#define DT_WAIT_BUDGET (1ll << 31)

// ---------------------------------------------------------------------------
// Element access and order-preserving keys.  A key is an unsigned integer
// whose order equals the numeric order of the value; -0 is mapped onto +0 so
// that equal values have equal keys.
// ---------------------------------------------------------------------------
template <typename T>
struct DtElem;

template <>
struct DtElem<uint16_t> {  // bf16 stored as raw bits
    static constexpr int KB = 16;
    static DT_DI float val(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }
    static DT_DI uint32_t key(uint16_t h) {
        if ((h & 0x7FFFu) == 0) h = 0;
        return (h & 0x8000u) ? (~uint32_t(h) & 0xFFFFu) : (uint32_t(h) | 0x8000u);
    }
    static DT_DI float key_val(uint32_t k) {
        uint32_t h = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
        return __uint_as_float(h << 16);
    }
};

template <>
struct DtElem<float> {
    static constexpr int KB = 32;
    static DT_DI float val(float x) { return x; }
    static DT_DI uint32_t key(float x) {
        uint32_t b = __float_as_uint(x);
        if ((b & 0x7FFFFFFFu) == 0) b = 0;
        return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    }
    static DT_DI float key_val(uint32_t k) {
        uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
        return __uint_as_float(b);
    }
};

// Order key of an fp32 score (same mapping as DtElem<float>).
DT_DI uint32_t dt_fkey(float x) { return DtElem<float>::key(x); }
DT_DI float dt_fkey_val(uint32_t k) { return DtElem<float>::key_val(k); }

// ---------------------------------------------------------------------------
// Warp / block reductions and scans.
// ---------------------------------------------------------------------------
DT_DI float dt_warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
DT_DI uint32_t dt_warp_max_u32(uint32_t v) {
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
DT_DI float dt_warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
DT_DI int dt_warp_sum_i(int v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
DT_DI unsigned long long dt_warp_sum_u64(unsigned long long v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
DT_DI int dt_warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Exclusive prefix sum of one int per thread over the block; returns the
// thread's exclusive prefix and writes the block total to *total.
// `red` needs NT/32 ints of shared memory.  Contains two __syncthreads.
template <int NT>
DT_DI int dt_block_excl_scan(int v, int* red, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int inc = dt_warp_incl_scan(v);
    if (lane == 31) red[w] = inc;
    __syncthreads();
    int wsum = (lane < NT / 32) ? red[lane] : 0;
    int winc = dt_warp_incl_scan(wsum);
    int before = __shfl_sync(0xffffffffu, winc, w) - __shfl_sync(0xffffffffu, wsum, w);
    int tot = __shfl_sync(0xffffffffu, winc, NT / 32 - 1);
    __syncthreads();
    *total = tot;
    return before + inc - v;
}

// Exclusive scan of an int array in shared memory (n entries, any n):
// out[i] = sum of a[0..i), out[n] = total.  in and out may alias.
template <int NT>
DT_DI void dt_block_scan_array(const int* a, int* out, int n, int* red) {
    int carry = 0;
    for (int base = 0; base < n; base += NT) {
        int i = base + threadIdx.x;
        int v = (i < n) ? a[i] : 0;
        int tot;
        int ex = dt_block_excl_scan<NT>(v, red, &tot);
        if (i < n) out[i] = carry + ex;
        carry += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) out[n] = carry;
    __syncthreads();
}

// In-place bitonic sort of n (a power of two) 64-bit keys in shared memory,
// descending when desc, else ascending.  Ends with __syncthreads.
template <int NT>
DT_DI void dt_bitonic_u64(unsigned long long* a, int n, bool desc) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += NT) {
                int ixj = i ^ j;
                if (ixj > i) {
                    unsigned long long x = a[i], y = a[ixj];
                    bool up = ((i & k) == 0) == desc;  // true: larger first
                    if (up ? (x < y) : (x > y)) { a[i] = y; a[ixj] = x; }
                }
            }
            __syncthreads();
        }
    }
}

// Sort n <= 32 64-bit keys in shared memory with warp 0 only (shuffles, no
// block barriers inside); descending when desc.  Ends with __syncthreads.
DT_DI void dt_warp_sort_u64(unsigned long long* a, int n, bool desc) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        // pad: sorts after every real key
        unsigned long long x = (lane < n) ? a[lane] : (desc ? 0ull : ~0ull);
        for (int k = 2; k <= 32; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
                const bool lower = (lane & j) == 0;
                const bool up = ((lane & k) == 0) == desc;  // larger first in this run
                const bool take_max = (lower == up);
                x = take_max ? (x > y ? x : y) : (x < y ? x : y);
            }
        }
        if (lane < n) a[lane] = x;
    }
    __syncthreads();
}

// Register-level warp sorts of one 64-bit key per lane (bitonic network on
// shuffles, no block barrier).  dt_warp_sort_reg: any order in, sorted out
// (descending when desc); dt_warp_merge_reg: a bitonic sequence in, sorted out.
DT_DI unsigned long long dt_warp_sort_reg(unsigned long long x, bool desc) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
            const bool take_max = (((lane & j) == 0) == (((lane & k) == 0) == desc));
            x = take_max ? (x > y ? x : y) : (x < y ? x : y);
        }
    }
    return x;
}
DT_DI unsigned long long dt_warp_merge_reg(unsigned long long x, bool desc) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
        const bool take_max = (((lane & j) == 0) == desc);
        x = take_max ? (x > y ? x : y) : (x < y ? x : y);
    }
    return x;
}
// Sort n <= 512 distinct 64-bit keys in shared memory (descending when desc)
// with two block barriers: warps sort 32-key segments in registers; a key's
// place is then its place in its segment plus, for each other segment, how
// many keys there come before it (a binary search over 32).  scratch:
// 32 * ceil(n / 32) keys, not overlapping a[0, n).  Pads (0 when desc, all
// ones otherwise) must not be valid keys.  Ends with __syncthreads.
template <int NT>
DT_DI void dt_block_sort_u64(unsigned long long* a, int n, bool desc, unsigned long long* scratch) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nseg = (n + 31) >> 5;
    for (int sg = wid; sg < nseg; sg += NT / 32) {
        const int i = sg * 32 + lane;
        const unsigned long long x = i < n ? a[i] : (desc ? 0ull : ~0ull);
        scratch[i] = dt_warp_sort_reg(x, desc);
    }
    __syncthreads();
    for (int i = tid; i < n; i += NT) {  // the pads sort to the end of the last segment
        const unsigned long long x = scratch[i];
        const int own = i >> 5;
        int rank = i & 31;
        for (int t = 0; t < nseg; ++t) {
            if (t == own) continue;
            const unsigned long long* seg = scratch + 32 * t;
            int lo = 0, hi = 32;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const unsigned long long y = seg[mid];
                if (desc ? (y > x) : (y < x)) lo = mid + 1;
                else hi = mid;
            }
            rank += lo;
        }
        a[rank] = x;
    }
    __syncthreads();
}

// a, b: descending warp lists (one key per lane).  Returns the 32 largest of
// their union, descending: the lane-wise maximum of a and reversed b is a
// bitonic sequence holding exactly those.
DT_DI unsigned long long dt_warp_top32_merge(unsigned long long a, unsigned long long b) {
    const unsigned long long r = __shfl_sync(0xffffffffu, b, 31 - (threadIdx.x & 31));
    return dt_warp_merge_reg(a > r ? a : r, true);
}

// The 32 largest of m keys key_of(0..m-1) (all nonzero), descending, one per
// lane of warp 0 (0 past the m-th); other warps get no result.  Each warp
// keeps a running top-32 over chunks of 32 keys, then the warps' lists merge
// pairwise in a tree through `scratch` (NT 64-bit words).  Must be called by
// all threads; contains log2(NT/32) __syncthreads and ends with one.
template <int NT, typename KeyFn>
DT_DI unsigned long long dt_block_top32(int m, KeyFn key_of, unsigned long long* scratch) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    constexpr int NW = NT / 32;
    unsigned long long R = 0ull;
    for (int base = wid * 32; base < m; base += NT) {
        const unsigned long long x = (base + lane < m) ? key_of(base + lane) : 0ull;
        R = dt_warp_top32_merge(R, dt_warp_sort_reg(x, true));
    }
#pragma unroll
    for (int lev = 1; lev < NW; lev <<= 1) {
        if ((wid & (2 * lev - 1)) == lev) scratch[wid * 32 + lane] = R;
        __syncthreads();
        if ((wid & (2 * lev - 1)) == 0 && wid + lev < NW) R = dt_warp_top32_merge(R, scratch[(wid + lev) * 32 + lane]);
    }
    __syncthreads();
    return R;
}

DT_DI int dt_pow2_ceil(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (TMA, 1-D) helpers.
// ---------------------------------------------------------------------------
DT_DI uint32_t dt_smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

DT_DI void dt_mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(dt_smem_addr(bar)), "r"(count) : "memory");
}
DT_DI void dt_fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
DT_DI void dt_fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
DT_DI void dt_mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(dt_smem_addr(bar)), "r"(bytes)
                 : "memory");
}
// Bulk copy global -> own shared memory; dst, src 16-byte aligned, bytes a multiple of 16.
DT_DI void dt_bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dt_smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(dt_smem_addr(bar))
        : "memory");
}
// Wait for the phase with parity `phase` to complete; false once `budget`
// SM clock cycles have passed without it.
DT_DI bool dt_mbar_wait_budget(uint64_t* bar, uint32_t phase, long long budget) {
    const uint32_t a = dt_smem_addr(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        // the hint lets the hardware suspend the thread until the phase
        // completes (up to ~10 ms) instead of returning at once, so waiting
        // warps do not take issue slots from co-resident work
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(phase), "r"(10000000u)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > budget) return false;
    }
}
DT_DI bool dt_mbar_wait(uint64_t* bar, uint32_t phase) { return dt_mbar_wait_budget(bar, phase, DT_WAIT_BUDGET); }

// Test hook of the timeout path (dt_test_wait_fault): a kernel whose probe
// budget is positive first waits, with that budget, on `probe` -- a barrier
// initialised with one expected arrival that nothing ever arrives on -- so the
// wait runs out and the kernel takes its timeout path; the real wait follows
// unchanged, so every copy still lands before the data is read.  Returns false
// when the probe ran out.
DT_DI bool dt_probe_wait(uint64_t* probe, long long budget) {
    return budget <= 0 || dt_mbar_wait_budget(probe, 0, budget);
}

// Programmatic dependent launch: every kernel of the library is launched so
// that it may start while the previous kernel in the stream is finishing.
// dt_pdl_wait() blocks until all prerequisite grids have completed and their
// memory is visible -- it must precede the first read of any input;
// dt_pdl_trigger() lets the next kernel in the stream be scheduled.
DT_DI void dt_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DT_DI void dt_pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Split cluster barrier: arrive (releasing this thread's prior shared-memory
// accesses) now, wait (acquiring every cluster thread's) later, so that local
// work can run in between.  Every thread of every CTA must execute both.
DT_DI void dt_cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
DT_DI void dt_cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// Packed fp32 pairs (one 64-bit register pair) for the two-lane f32x2
// instructions; every operation is rounded to nearest on its own.
DT_DI unsigned long long dt_f2_pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
DT_DI void dt_f2_unpack(unsigned long long r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
DT_DI unsigned long long dt_f2_sub(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
DT_DI unsigned long long dt_f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
DT_DI unsigned long long dt_f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
DT_DI unsigned long long dt_f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ---------------------------------------------------------------------------
// 16-byte vectors of staged row elements (8 bf16 or 4 fp32).
// ---------------------------------------------------------------------------
// Hardware base-2 exponential (approximate, ~2 ulp); used only for
// log-normaliser sums, whose tolerance is 1e-5.
DT_DI float dt_ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The element type's bits of a value that came from that type (exact).
template <typename T> DT_DI T dt_to_elem(float x);
template <> DT_DI uint16_t dt_to_elem<uint16_t>(float x) { return (uint16_t)(__float_as_uint(x) >> 16); }
template <> DT_DI float dt_to_elem<float>(float x) { return x; }

// Values of the elements of a 16-byte vector, as fp32.
template <typename T> DT_DI void dt_vec_vals(const uint4& q, float (&x)[16 / sizeof(T)]);
template <> DT_DI void dt_vec_vals<uint16_t>(const uint4& q, float (&x)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}
template <> DT_DI void dt_vec_vals<float>(const uint4& q, float (&x)[4]) {
    x[0] = __uint_as_float(q.x);
    x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z);
    x[3] = __uint_as_float(q.w);
}

// Largest value of a full 16-byte vector (bf16: packed two-way compares).
template <typename T> DT_DI float dt_vec_max(const uint4& q);
template <> DT_DI float dt_vec_max<uint16_t>(const uint4& q) {
    const __nv_bfloat162 a = __hmax2(*(const __nv_bfloat162*)&q.x, *(const __nv_bfloat162*)&q.y);
    const __nv_bfloat162 b = __hmax2(*(const __nv_bfloat162*)&q.z, *(const __nv_bfloat162*)&q.w);
    const __nv_bfloat162 c = __hmax2(a, b);
    return fmaxf(__low2float(c), __high2float(c));
}
template <> DT_DI float dt_vec_max<float>(const uint4& q) {
    return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)), fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
}

// acc + (exp2((x0 - m) * log2e), exp2((x1 - m) * log2e)), two lanes at once;
// m2 and l2 hold (m, m) and (log2e, log2e).  The difference is rounded before
// the product, so x = m gives exactly 1 at any magnitude.
DT_DI unsigned long long dt_pair_exp(float x0, float x1, unsigned long long m2, unsigned long long l2,
                                     unsigned long long acc) {
    float d0, d1;
    dt_f2_unpack(dt_f2_mul(dt_f2_sub(dt_f2_pack(x0, x1), m2), l2), d0, d1);
    return dt_f2_add(acc, dt_f2_pack(dt_ex2_approx(d0), dt_ex2_approx(d1)));
}
// acc + the pairwise exp sums of every element of a full vector.
template <typename T> DT_DI unsigned long long dt_vec_expsum(const uint4& q, unsigned long long m2,
                                                           unsigned long long l2, unsigned long long acc);
template <> DT_DI unsigned long long dt_vec_expsum<uint16_t>(const uint4& q, unsigned long long m2,
                                                           unsigned long long l2, unsigned long long acc) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        acc = dt_pair_exp(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u), m2, l2, acc);
    return acc;
}
template <> DT_DI unsigned long long dt_vec_expsum<float>(const uint4& q, unsigned long long m2,
                                                        unsigned long long l2, unsigned long long acc) {
    acc = dt_pair_exp(__uint_as_float(q.x), __uint_as_float(q.y), m2, l2, acc);
    return dt_pair_exp(__uint_as_float(q.z), __uint_as_float(q.w), m2, l2, acc);
}

// Stage elements [lo, hi) of a row into shared memory.  The shared buffer
// `sbase` must be 16-byte aligned with room for (hi - lo) elements + 16 bytes;
// the returned pointer is where element lo lands (sbase + (src address mod 16)).
// The 16-byte-aligned interior moves with one bulk copy completing on `bar`
// (one elected thread issues it); the ragged head and tail use plain loads by
// all threads.  Returns the number of bytes the bulk copy will deliver (0 if
// none) -- the caller waits on `bar` for that phase when it is non-zero.
// Must be called by all threads of the block.
template <typename T>
DT_DI const T* dt_stage_row(const T* row, int lo, int hi, unsigned char* sbase, uint64_t* bar,
                            uint32_t* bulk_bytes) {
    const uintptr_t a_lo = (uintptr_t)(row + lo);
    const uintptr_t a_hi = (uintptr_t)(row + hi);
    T* s = (T*)(sbase + (a_lo & 15));
    uintptr_t in_lo = (a_lo + 15) & ~(uintptr_t)15;
    uintptr_t in_hi = a_hi & ~(uintptr_t)15;
    uint32_t bytes = 0;
    if (in_hi > in_lo) bytes = (uint32_t)(in_hi - in_lo);
    else { in_lo = a_hi; in_hi = a_hi; }
    const int e_in_lo = (int)((in_lo - a_lo) / sizeof(T));
    const int e_in_hi = (int)((in_hi - a_lo) / sizeof(T));
    const int n = hi - lo;
    if (threadIdx.x == 0 && bytes) {
        dt_mbar_arrive_expect_tx(bar, bytes);
        dt_bulk_g2s(s + e_in_lo, (const void*)in_lo, bytes, bar);
    }
    for (int e = threadIdx.x; e < e_in_lo; e += blockDim.x) s[e] = row[lo + e];
    for (int e = e_in_hi + threadIdx.x; e < n; e += blockDim.x) s[e] = row[lo + e];
    *bulk_bytes = bytes;
    return s;
}

// Per-thread asynchronous 16-byte copies global -> shared (L2 only, not L1),
// grouped: commit closes a group; wait<N> returns once at most N of this
// thread's groups are still in flight.
DT_DI void dt_cp_async16(void* sdst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dt_smem_addr(sdst)), "l"(gsrc) : "memory");
}
DT_DI void dt_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Copies the first src_bytes (0..16) of 16 bytes and zero-fills the rest.
DT_DI void dt_cp_async16_zfill(void* sdst, const void* gsrc, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dt_smem_addr(sdst)), "l"(gsrc), "r"(src_bytes)
                 : "memory");
}
// Arrives on the mbarrier once all of this thread's earlier cp.async copies
// have landed (the arrival is counted in the barrier's expected count).
DT_DI void dt_cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(dt_smem_addr(bar)) : "memory");
}
// Plain mbarrier arrival by this thread.
DT_DI void dt_mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(dt_smem_addr(bar)) : "memory");
}
template <int N>
DT_DI void dt_cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Chunk staging in two steps, for prefetching.  start(): one thread issues the
// bulk copy of the 16-byte-aligned interior of elements [lo, hi) of `row`
// (completing on `bar`), and the ragged head and tail elements (fewer than 16
// of each) are loaded into registers of threads 0-15 and 16-31; it returns the
// bulk bytes (0: nothing to wait for on `bar`).  finish(): those threads store
// their element into the buffer; the caller syncs the block before reading.
// The load latency of the ragged elements thus overlaps whatever runs between
// the two calls.  Element lo lands at sbase + (address of row + lo) mod 16, as
// with dt_stage_row.  Both must be called by all threads of the block.
template <typename T>
struct DtStager {
    T held;
    int held_off;  // byte offset of the held element in the buffer; -1: none

    DT_DI uint32_t start(const T* row, int lo, int hi, unsigned char* sbase, uint64_t* bar) {
        const uintptr_t a_lo = (uintptr_t)(row + lo);
        const uintptr_t a_hi = (uintptr_t)(row + hi);
        const int off0 = (int)(a_lo & 15);
        uintptr_t in_lo = (a_lo + 15) & ~(uintptr_t)15;
        uintptr_t in_hi = a_hi & ~(uintptr_t)15;
        uint32_t bytes = 0;
        if (in_hi > in_lo) bytes = (uint32_t)(in_hi - in_lo);
        else { in_lo = a_hi; in_hi = a_hi; }  // no aligned interior: fewer than 32 bytes in all
        const int e_in_lo = (int)((in_lo - a_lo) / sizeof(T));
        const int e_in_hi = (int)((in_hi - a_lo) / sizeof(T));
        const int n = hi - lo;
        if (threadIdx.x == 0 && bytes) {
            dt_mbar_arrive_expect_tx(bar, bytes);
            dt_bulk_g2s(sbase + off0 + (size_t)e_in_lo * sizeof(T), (const void*)in_lo, bytes, bar);
        }
        const int t = threadIdx.x;
        int e = -1;
        if (t < 16) {
            if (t < e_in_lo) e = t;
        } else if (t < 32) {
            if (e_in_hi + (t - 16) < n) e = e_in_hi + (t - 16);
        }
        held_off = -1;
        if (e >= 0) {
            held = row[lo + e];
            held_off = off0 + e * (int)sizeof(T);
        }
        return bytes;
    }
    DT_DI void finish(unsigned char* sbase) const {
        if (held_off >= 0) *(T*)(sbase + held_off) = held;
    }
};

// ---------------------------------------------------------------------------
// Shared node order on explicit node arrays (score s, depth dep, parent par,
// lex = (lexicographic rank of the parent among its depth << 16) | own rank):
// does node y come before node x?  Higher score first; on equal scores the
// lexicographically smaller rank descriptor, a prefix before its extensions.
// Nodes of the same depth compare by lex; otherwise the deeper node is walked
// up to the shallower one's depth.
// ---------------------------------------------------------------------------
DT_DI bool dt_node_before(int y, int x, const float* s, const int* dep, const int* par, const uint32_t* lex) {
    const float sy = s[y], sx = s[x];
    if (sy != sx) return sy > sx;
    const int dy = dep[y], dx = dep[x];
    if (dy == dx) return lex[y] < lex[x];
    if (dy < dx) {
        int a = x;
        while (dep[a] > dy) a = par[a];
        if (a == y) return true;
        return lex[y] < lex[a];
    }
    int a = y;
    while (dep[a] > dx) a = par[a];
    if (a == x) return false;
    return lex[a] < lex[x];
}

// Bitonic sort of n (a power of two) node indices by dt_node_before; entries
// equal to -1 are padding and sort last.  Ends with __syncthreads.
template <int NT>
DT_DI void dt_bitonic_nodes(int* a, int n, const float* s, const int* dep, const int* par, const uint32_t* lex) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += NT) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const int x = a[i], y = a[ixj];
                    // does y belong before x?
                    bool y_first;
                    if (x < 0) y_first = (y >= 0);
                    else if (y < 0) y_first = false;
                    else y_first = dt_node_before(y, x, s, dep, par, lex);
                    const bool asc = ((i & k) == 0);
                    if (asc ? y_first : (!y_first && x != y)) { a[i] = y; a[ixj] = x; }
                }
            }
            __syncthreads();
        }
    }
}
