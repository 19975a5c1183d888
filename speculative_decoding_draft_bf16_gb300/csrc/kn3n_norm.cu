// kn3n_norm.cu -- full-vocabulary log-normalisers of the corrected DARTree
// drafter distribution, on the tensor cores.
//
// [DARTree] "Causal correction": the corrected distribution q~ is a
// probability over the vocabulary, q~_d(v | u) = exp(lp_d(v) + <U[u], Vt[v]>)
// / Z_d(u).  Row (b, d, i) of the table holds log Z_d(u) for the parent token
// u of request b's depth-(d+1) children: the i-th candidate of position d-1,
// or the root token at d = 0 (row i = 0 only); rows without a parent token
// hold 0.
//
// log Z_d(u) = logsumexp_v (x_d(v) + <U[u], Vt[v]>) - lse_d.  The [rows x R]
// x [R x V] contraction (R = 64) is the one dense contraction of the method:
// it runs on the fifth-generation tensor cores (tcgen05.mma, kind::f16, fp32
// accumulation in tensor memory).  The tables are fp32; each is split into a
// bf16 head and a bf16 tail (U = Uh + Ul + e with |e| <= 2^-18 |U|, the tail
// being the rounded remainder), and the accumulator takes all four products
// Uh.Vh + Uh.Vl + Ul.Vh + Ul.Vl (products of bf16 values are exact in fp32),
// so each dot product is within about 2^-17 * sum_k |U_k Vt_k| of the fp32
// tables' -- the bf16 rounding of a single product would leave 2^-8.
// Each CTA takes a tile of 128 rows and a slice of the vocabulary: it stages
// the rows' U vectors once (head and tail, 128-byte-swizzled K-major bf16
// tiles) and, per 128-token step, the tokens' Vt tiles -- laid out in global
// memory by the conversion kernel exactly as the tensor cores read them, so
// one 32 KB bulk copy brings a step's head and tail -- issues sixteen
// 128x128x16 MMAs from one thread, and its eight epilogue warps read the
// 128x128 fp32 accumulator back, add the drafter logits and fold exp into a
// running (max, sum) per row.  A second kernel merges the slices.
#include <cuda_bf16.h>

#include "dt_launch.h"
#include "dt_tcgen05.cuh"

namespace {

constexpr int NT = 320;       // warps 0-7: epilogue; warp 8: copies; warp 9: MMA issue
constexpr int NEPI = 256;     // epilogue threads: TMEM lane quarter (warp % 4) x column half (warp / 4)
constexpr int STAGES = 2;     // ring of Vt / logit tiles
constexpr int TM = 128;       // rows per tile
constexpr int TN = 128;       // tokens per MMA step
constexpr int RK = 64;        // contraction length R (64 bf16 = one 128-byte row)
constexpr int XG = 16;        // (request, position) logit rows staged per step, at most
constexpr uint32_t IDESC = dt_idesc_bf16_f32(TM, TN);
constexpr size_t HALF = 16384;                            // one 128 x 64 bf16 tile
constexpr size_t A_BYTES = 2 * HALF, B_BYTES = 2 * HALF;  // head tile, then tail tile
constexpr size_t X_BYTES = (size_t)XG * TN * 2;           // bf16 logit rows (fp32 logits are read in place)
constexpr size_t OFF_B = A_BYTES;
constexpr size_t OFF_X = OFF_B + STAGES * B_BYTES;
constexpr size_t OFF_BAR = OFF_X + STAGES * X_BYTES;

struct Kn3nShared {
    uint64_t full[STAGES];   // tile landed (the Vt bulk copy + 32 logit-copy arrivals)
    uint64_t empty[STAGES];  // tile consumed (MMA commit + NEPI logit readers)
    uint64_t accf[2];        // accumulator written (MMA commit)
    uint64_t acce[2];        // accumulator read (NEPI arrivals)
    uint64_t probe;          // the timeout-path test hook's barrier (never completes)
    uint32_t tmem;
    int fail;
    float pm[TM], ps[TM];    // second column half's partial (max, sum) per row
};
// The A tiles, two B stages and two logit tiles from a 1024-byte aligned base;
// at most two CTAs fit an SM, so their 2 x 256 TMEM columns always fit its 512
constexpr size_t SMEM = 1024 + OFF_BAR + sizeof(Kn3nShared);
static_assert(2 * (SMEM + 1024) <= 233472 && 3 * (SMEM + 1024) > 233472, "two CTAs per SM, not three");

// Parent token of row r (-1: the row has no term).
DT_DI int row_parent(int r, int L, int K, int V, const int32_t* root_tok, const int32_t* cand_id, int* b, int* d) {
    *b = r / (L * K);
    *d = (r / K) % L;
    const int i = r % K;
    int u;
    if (*d == 0) u = (i == 0 && root_tok) ? root_tok[*b] : -1;
    else u = cand_id[((size_t)*b * L + *d - 1) * K + i];
    return (u >= 0 && u < V) ? u : -1;
}

// bf16 head and tail of two fp32 values (round to nearest; the tail is the
// rounded remainder, which fp32 holds exactly).
DT_DI void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(__fsub_rn(a, hf.x), __fsub_rn(b, hf.y));
    hi = *(const uint32_t*)&h;
    lo = *(const uint32_t*)&l;
}

// Columns [k0, k0 + 32) of an fp32 [*, 64] table row into the swizzled bf16
// head tile and tail tile (HALF bytes after it); zeros when src is null.
DT_DI void stage_half_row_split(unsigned char* tile, int row, int k0, const float* src) {
#pragma unroll
    for (int k = k0; k < k0 + 32; k += 4) {
        float4 f = src ? *(const float4*)(src + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        uint2 wh, wl;
        split2(f.x, f.y, wh.x, wl.x);
        split2(f.z, f.w, wh.y, wl.y);
        *(uint2*)(tile + dt_sw128_offset(row, k)) = wh;
        *(uint2*)(tile + HALF + dt_sw128_offset(row, k)) = wl;
    }
}

// Bounded wait; records a timeout in *fail (outputs then become NaN).
DT_DI void wait_or_fail(uint64_t* bar, uint32_t parity, int* fail) {
    if (!dt_mbar_wait(bar, parity)) *fail = 1;
}

// Fp32 Vt [V][64] -> per 128-token tile a 32 KB block [head | tail], each
// half the K-major 128-byte-swizzled bf16 layout the MMA reads (row r's
// 16-byte chunk c at r * 128 + ((c ^ (r % 8)) << 4)); rows past V are zero.
// One thread per (token, chunk of 8 values).
__global__ void __launch_bounds__(256) kn3n_convert_kernel(const float* __restrict__ src, unsigned char* __restrict__ dst,
                                                           int V, int ntiles) {
    dt_pdl_trigger();
    dt_pdl_wait();
    const size_t n = (size_t)ntiles * TN * 8;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int v = (int)(i >> 3), c = (int)(i & 7);
        const int t = v / TN, r = v % TN;
        uint4 wh = make_uint4(0u, 0u, 0u, 0u), wl = wh;
        if (v < V) {
            const float4 a = ((const float4*)(src + (size_t)v * RK + c * 8))[0];
            const float4 b = ((const float4*)(src + (size_t)v * RK + c * 8))[1];
            split2(a.x, a.y, wh.x, wl.x);
            split2(a.z, a.w, wh.y, wl.y);
            split2(b.x, b.y, wh.z, wl.z);
            split2(b.z, b.w, wh.w, wl.w);
        }
        unsigned char* base = dst + (size_t)t * B_BYTES + (size_t)r * 128 + ((c ^ (r & 7)) << 4);
        *(uint4*)base = wh;
        *(uint4*)(base + HALF) = wl;
    }
}

// The 32 logits of this thread's chunk from the staged tile, as fp32.
DT_DI void tile_x32(const uint16_t* xt, float (&o)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float t[8];
        dt_vec_vals<uint16_t>(*(const uint4*)(xt + 8 * q), t);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[8 * q + i] = t[i];
    }
}
DT_DI void tile_x32(const float* xt, float (&o)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float t[4];
        dt_vec_vals<float>(*(const uint4*)(xt + 4 * q), t);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[4 * q + i] = t[i];
    }
}

// Folds v[0..31] (entries from nvalid on excluded) into a running (max M,
// sum S of exp(v - M)).  For |M| < 64 each term is exp2(v * log2e - c) with
// c = M * log2e rounded, one fused multiply-add on two lanes at a time: c's
// rounding error (<= 2^-18) is common to every term of the row and shifts
// log Z by < 3e-6.  Larger maxima round v - M first.
DT_DI void fold32(float (&v)[32], int nvalid, float& M, float& S) {
    const float NEG_INF = -__int_as_float(0x7F800000);
    const float log2e = 1.44269504088896340736f;
    if (nvalid < 32) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i >= nvalid) v[i] = NEG_INF;
    }
    float cm = v[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) cm = fmaxf(cm, v[i]);
    if (cm > M) {
        S = (M == NEG_INF) ? 0.f : __fmul_rn(S, dt_ex2_approx(__fmul_rn(__fsub_rn(M, cm), log2e)));
        M = cm;
    }
    if (M == NEG_INF) return;
    if (fabsf(M) < 64.f) {
        const float c = __fmul_rn(M, log2e);
        const unsigned long long l2 = dt_f2_pack(log2e, log2e), c2 = dt_f2_pack(-c, -c);
        unsigned long long acc = dt_f2_pack(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            float d0, d1;
            dt_f2_unpack(dt_f2_fma(dt_f2_pack(v[i], v[i + 1]), l2, c2), d0, d1);
            acc = dt_f2_add(acc, dt_f2_pack(dt_ex2_approx(d0), dt_ex2_approx(d1)));
        }
        float a0, a1;
        dt_f2_unpack(acc, a0, a1);
        S = __fadd_rn(S, __fadd_rn(a0, a1));
    } else {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) p = __fadd_rn(p, dt_ex2_approx(__fmul_rn(__fsub_rn(v[i], M), log2e)));
        S = __fadd_rn(S, p);
    }
}

// Probe budget of the timeout-path test hook (0: off), set by dt_kn3n_set_probe.
__device__ long long g_kn3n_probe;

template <typename T>
__global__ void __launch_bounds__(NT, 2) kn3n_kernel(const T* __restrict__ x, int V, int L, int K, int rows,
                                                     const int32_t* __restrict__ root_tok,
                                                     const int32_t* __restrict__ cand_id,
                                                     const float* __restrict__ U, const unsigned char* __restrict__ Vtt,
                                                     int vs, float2* __restrict__ part) {
    using E = DtElem<T>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Kn3nShared* sh = (Kn3nShared*)(sm + OFF_BAR);
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, tile = blockIdx.y;
    const int vbeg = split * vs, vend = min(V, vbeg + vs);
    const int nsteps = (vend - vbeg + TN - 1) / TN;
    const float NEG_INF = -__int_as_float(0x7F800000);
    const float log2e = 1.44269504088896340736f;
    // logit rows of this tile: flat (request, position) indices g0 .. g0 + ng - 1
    const int g0 = (tile * TM) / K;
    const int ng = (min(rows, tile * TM + TM) - 1) / K - g0 + 1;
    const bool xs = sizeof(T) == 2 && ng <= XG && (((uintptr_t)x) & 15u) == 0 && ((size_t)V * sizeof(T)) % 16 == 0;

    if (wid == 0) dt_tmem_alloc(&sh->tmem, 2 * TN);
    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            dt_mbar_init(&sh->full[i], 33);
            dt_mbar_init(&sh->empty[i], 1 + NEPI);
        }
        for (int i = 0; i < 2; ++i) {
            dt_mbar_init(&sh->accf[i], 1);
            dt_mbar_init(&sh->acce[i], NEPI);
        }
        dt_mbar_init(&sh->probe, 1);
        dt_fence_mbar_init();
        sh->fail = 0;
    }
    dt_pdl_trigger();
    dt_pdl_wait();  // candidate ids, logits and the bf16 table come from earlier kernels

    if (tid < NEPI) {  // A tiles: the rows' U vectors (head, tail), two threads per row
        const int row = tid & (TM - 1), r = tile * TM + row;
        int b, d;
        const int u = r < rows ? row_parent(r, L, K, V, root_tok, cand_id, &b, &d) : -1;
        stage_half_row_split(sm, row, 32 * (tid >> 7), u >= 0 ? U + (size_t)u * RK : nullptr);
    }
    dt_fence_proxy_async_smem();
    dt_tc_fence_before();
    __syncthreads();
    dt_tc_fence_after();
    const uint32_t tmem = sh->tmem;

    if (wid == 8) {
        // ---- copies: the step's Vt tile pair (one bulk copy) and logit rows
        for (int j = 0; j < nsteps; ++j) {
            const int s = j % STAGES;
            if (j >= STAGES) wait_or_fail(&sh->empty[s], ((j / STAGES) - 1) & 1, &sh->fail);
            const int v0 = vbeg + j * TN;
            if (lane == 0) {
                dt_mbar_arrive_expect_tx(&sh->full[s], (uint32_t)B_BYTES);
                dt_bulk_g2s(sm + OFF_B + s * B_BYTES, Vtt + (size_t)(v0 / TN) * B_BYTES, (uint32_t)B_BYTES,
                            &sh->full[s]);
            }
            if constexpr (sizeof(T) == 2) if (xs) {
                constexpr int EPC = 16 / sizeof(T);   // elements per 16-byte chunk
                constexpr int CPR = TN / EPC;         // chunks per logit row
                unsigned char* xt = sm + OFF_X + s * X_BYTES;
                for (int q = lane; q < ng * CPR; q += 32) {
                    const int g = q / CPR, c = q % CPR, e0 = v0 + c * EPC;
                    const int nb = max(0, min(16, (vend - e0) * (int)sizeof(T)));
                    const T* src = x + (size_t)(g0 + g) * V + e0;
                    dt_cp_async16_zfill(xt + (size_t)g * TN * sizeof(T) + c * 16, nb > 0 ? (const void*)src : (const void*)x,
                                        (uint32_t)nb);
                }
            }
            dt_cp_async_arrive(&sh->full[s]);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (wid == 9) {
        // ---- MMA issue: 128 x 128 x 64 per step into alternating accumulators
        if (lane == 0) {
            const uint32_t ab = dt_smem_addr(sm);
            if (!dt_probe_wait(&sh->probe, g_kn3n_probe)) sh->fail = 1;
            for (int j = 0; j < nsteps; ++j) {
                const int s = j % STAGES, a = j & 1;
                wait_or_fail(&sh->full[s], (j / STAGES) & 1, &sh->fail);
                if (j >= 2) wait_or_fail(&sh->acce[a], ((j >> 1) - 1) & 1, &sh->fail);
                dt_tc_fence_after();
                dt_fence_proxy_async_smem();
                const uint32_t bb = dt_smem_addr(sm + OFF_B + s * B_BYTES);
                // head x head, then the three products with a tail
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
                    const uint32_t ao = ab + (pr >> 1) * (uint32_t)HALF, bo = bb + (pr & 1) * (uint32_t)HALF;
#pragma unroll
                    for (int kk = 0; kk < RK / 16; ++kk)
                        dt_mma_bf16(tmem + a * TN, dt_desc_kmajor_sw128(ao + 32 * kk),
                                    dt_desc_kmajor_sw128(bo + 32 * kk), IDESC, pr > 0 || kk > 0);
                }
                dt_mma_commit(&sh->empty[s]);
                dt_mma_commit(&sh->accf[a]);
            }
        }
    }
    float m_run = NEG_INF, s_run = 0.f;
    const int q4 = wid & 3, h = wid >> 2;     // epilogue: lane quarter, column half
    const int row = q4 * 32 + lane, r = tile * TM + row;
    if (wid < 8) {
        // ---- epilogue: accumulator + logit, folded into a running (max, sum)
        int b = 0, d = 0;
        const int u = r < rows ? row_parent(r, L, K, V, root_tok, cand_id, &b, &d) : -1;
        const int g = u >= 0 ? (b * L + d) - g0 : 0;  // logit row within the staged tile
        const T* xrow = x + ((size_t)b * L + d) * V;
        for (int j = 0; j < nsteps; ++j) {
            const int s = j % STAGES, a = j & 1;
            const int c0 = vbeg + j * TN + h * 64;  // first token of this thread's columns
            const T* xt = (const T*)(sm + OFF_X + s * X_BYTES) + (size_t)g * TN + h * 64;
            wait_or_fail(&sh->accf[a], (j >> 1) & 1, &sh->fail);
            if (xs) wait_or_fail(&sh->full[s], (j / STAGES) & 1, &sh->fail);  // the logit tile has landed
            dt_tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(q4 * 32) << 16) + a * TN + h * 64;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float v[32];
                dt_tmem_ld32(ta + 32 * half, v);
                const int cb = c0 + 32 * half;             // token of v[0]
                const int nvalid = u >= 0 ? max(0, min(32, vend - cb)) : 0;
                if (nvalid > 0) {
                    float xv[32];
                    if (xs) {
                        tile_x32(xt + 32 * half, xv);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) xv[i] = (i < nvalid) ? E::val(xrow[cb + i]) : 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float a0, a1;
                        dt_f2_unpack(dt_f2_add(dt_f2_pack(v[i], v[i + 1]), dt_f2_pack(xv[i], xv[i + 1])), a0, a1);
                        v[i] = a0;
                        v[i + 1] = a1;
                    }
                }
                if (half == 1) {
                    dt_tc_fence_before();
                    dt_mbar_arrive(&sh->acce[a]);   // accumulator free for step j + 2
                    dt_mbar_arrive(&sh->empty[s]);  // logit tile read
                }
                if (nvalid > 0) fold32(v, nvalid, m_run, s_run);
            }
        }
        if (h == 1) {
            sh->pm[row] = m_run;
            sh->ps[row] = s_run;
        }
    }
    dt_tc_fence_before();
    __syncthreads();
    if (wid < 4 && r < rows) {
        // merge the two column halves; a bounded wait that ran out leaves NaN
        const float m2 = sh->pm[row], s2 = sh->ps[row];
        const float M = fmaxf(m_run, m2);
        float S = 0.f;
        if (m_run != NEG_INF) S = __fmul_rn(s_run, dt_ex2_approx(__fmul_rn(__fsub_rn(m_run, M), log2e)));
        if (m2 != NEG_INF) S = __fadd_rn(S, __fmul_rn(s2, dt_ex2_approx(__fmul_rn(__fsub_rn(m2, M), log2e))));
        part[(size_t)r * gridDim.x + split] = sh->fail ? make_float2(__int_as_float(0x7FC00000), 0.f) : make_float2(M, S);
    }
    if (wid == 0) {
        dt_tc_fence_after();
        dt_tmem_dealloc(tmem, 2 * TN);
    }
}

// log Z = max + log(sum) - lse per row, merging the vocabulary slices.
__global__ void __launch_bounds__(256) kn3n_reduce_kernel(const float2* __restrict__ part, int nsplit, int rows,
                                                          int L, int K, int V, const int32_t* __restrict__ root_tok,
                                                          const int32_t* __restrict__ cand_id,
                                                          const float* __restrict__ lse, float* __restrict__ z) {
    const float NEG_INF = -__int_as_float(0x7F800000);
    const float log2e = 1.44269504088896340736f;
    dt_pdl_trigger();
    dt_pdl_wait();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    int b, d;
    const int u = row_parent(r, L, K, V, root_tok, cand_id, &b, &d);
    if (u < 0) {
        z[r] = 0.f;
        return;
    }
    float M = NEG_INF;
    bool bad = false;
    for (int j = 0; j < nsplit; ++j) {
        const float mj = part[(size_t)r * nsplit + j].x;
        bad |= (mj != mj);
        M = fmaxf(M, mj);
    }
    if (bad) {
        z[r] = __int_as_float(0x7FC00000);  // the selection reports DT_DEV_TIMEOUT
        return;
    }
    float S = 0.f;
    for (int j = 0; j < nsplit; ++j) {
        const float2 p = part[(size_t)r * nsplit + j];
        if (p.x != NEG_INF) S = __fadd_rn(S, __fmul_rn(p.y, dt_ex2_approx(__fmul_rn(__fsub_rn(p.x, M), log2e))));
    }
    z[r] = __fsub_rn(__fadd_rn(M, logf(S)), lse[(size_t)b * L + d]);
}

}  // namespace

cudaError_t dt_kn3n_set_probe(long long budget) {
    return cudaMemcpyToSymbol(g_kn3n_probe, &budget, sizeof(budget));
}

size_t dt_kn3n_scratch_bytes(int rows, int V) {
    const size_t part = (((size_t)rows * DT_KN3N_MAX_SPLIT * sizeof(float2)) + 255) & ~(size_t)255;
    return part + (size_t)((V + TN - 1) / TN) * B_BYTES;
}

cudaError_t dt_kn3n_launch(const void* x, int dtype, int batch, int L, int K, int V, const int32_t* root_tok,
                           const int32_t* cand_id, const float* lse, const float* U, const float* Vt, void* scratch,
                           float* z, cudaStream_t st) {
    const int rows = batch * L * K;
    const int mtiles = (rows + TM - 1) / TM;
    float2* part = (float2*)scratch;
    unsigned char* Vtt = (unsigned char*)scratch +
                         ((((size_t)rows * DT_KN3N_MAX_SPLIT * sizeof(float2)) + 255) & ~(size_t)255);
    const int ntiles = (V + TN - 1) / TN;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms < 1) {
        (void)cudaGetLastError();
        sms = 148;
    }
    cudaError_t e;
    // the child-token table as bf16 head and tail tiles, once per call
    const size_t n8 = (size_t)ntiles * TN * 8;
    size_t cblocks = (n8 + 255) / 256;
    if (cblocks > (size_t)sms * 8) cblocks = (size_t)sms * 8;
    DtLaunch lcv(dim3((unsigned)cblocks), dim3(256), 0, st);
    if ((e = cudaLaunchKernelEx(&lcv.cfg, kn3n_convert_kernel, Vt, Vtt, V, ntiles)) != cudaSuccess) return e;
    // two CTAs per SM, vocabulary slices of whole 128-token steps
    int nsplit = (2 * sms + mtiles - 1) / mtiles;
    const int steps = (V + TN - 1) / TN;
    nsplit = max(1, min(min(nsplit, DT_KN3N_MAX_SPLIT), steps));
    const int vs = ((steps + nsplit - 1) / nsplit) * TN;
    nsplit = (V + vs - 1) / vs;
    DtLaunch lc(dim3(nsplit, mtiles, 1), dim3(NT, 1, 1), SMEM, st);
    if (dtype == DT_BF16) {
        if ((e = cudaFuncSetAttribute(kn3n_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) !=
            cudaSuccess)
            return e;
        e = cudaLaunchKernelEx(&lc.cfg, kn3n_kernel<uint16_t>, (const uint16_t*)x, V, L, K, rows, root_tok, cand_id, U,
                               (const unsigned char*)Vtt, vs, part);
    } else {
        if ((e = cudaFuncSetAttribute(kn3n_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) !=
            cudaSuccess)
            return e;
        e = cudaLaunchKernelEx(&lc.cfg, kn3n_kernel<float>, (const float*)x, V, L, K, rows, root_tok, cand_id, U,
                               (const unsigned char*)Vtt, vs, part);
    }
    if (e != cudaSuccess) return e;
    DtLaunch lr(dim3((rows + 255) / 256), dim3(256), 0, st);
    return cudaLaunchKernelEx(&lr.cfg, kn3n_reduce_kernel, (const float2*)part, nsplit, rows, L, K, V, root_tok,
                              cand_id, lse, z);
}
