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
// it runs on the fifth-generation tensor cores (tcgen05.mma, kind::f16, bf16
// operands rounded to nearest from the fp32 tables, fp32 accumulation in
// tensor memory).  Each CTA takes a tile of 128 rows and a slice of the
// vocabulary: it stages the rows' U vectors once and, per 128-token step, the
// tokens' Vt vectors (both as 128-byte-swizzled K-major bf16 tiles), issues
// four 128x128x16 MMAs from one thread, and its four warps read the 128x128
// fp32 accumulator back (one row per thread), add the drafter logits and fold
// exp into a running (max, sum) per row.  A second kernel merges the slices.
#include <cuda_bf16.h>

#include "dt_launch.h"
#include "dt_tcgen05.cuh"

namespace {

constexpr int NT = 128;       // four warps: TMEM lanes 0..127, one row each
constexpr int TM = 128;       // rows per tile
constexpr int TN = 128;       // tokens per MMA step
constexpr int RK = 64;        // contraction length R (64 bf16 = one 128-byte row)
constexpr uint32_t IDESC = dt_idesc_bf16_f32(TM, TN);
// alignment slack, A and B tiles, barrier; padded so that at most four CTAs
// share an SM, whose 512 TMEM columns then always cover their allocations
constexpr size_t SMEM = 56 * 1024;

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

// Row `row` of an fp32 [*, 64] table into an swizzled bf16 tile row (zeros when src is null).
DT_DI void stage_row_bf16(unsigned char* tile, int row, const float* src) {
#pragma unroll
    for (int k = 0; k < RK; k += 4) {
        float4 f = src ? *(const float4*)(src + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(f.x, f.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(f.z, f.w);
        uint2 w;
        w.x = *(const uint32_t*)&lo;
        w.y = *(const uint32_t*)&hi;
        *(uint2*)(tile + dt_sw128_offset(row, k)) = w;
    }
}

// 32 drafter logits x[v0 .. v0+31] as fp32 (-inf from vend on).
template <typename T>
DT_DI void load_x32(const T* xrow, int v0, int vend, float (&o)[32]) {
    using E = DtElem<T>;
    const float NEG_INF = -__int_as_float(0x7F800000);
    const T* p = xrow + v0;
    if (v0 + 32 <= vend && (((uintptr_t)p) & 15u) == 0) {
        constexpr int EPV = 16 / sizeof(T);
#pragma unroll
        for (int q = 0; q < 32 / EPV; ++q) {
            float t[EPV];
            dt_vec_vals<T>(*(const uint4*)(p + q * EPV), t);
#pragma unroll
            for (int s = 0; s < EPV; ++s) o[q * EPV + s] = t[s];
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = (v0 + j < vend) ? E::val(p[j]) : NEG_INF;
    }
}

template <typename T>
__global__ void __launch_bounds__(NT) kn3n_kernel(const T* __restrict__ x, int V, int L, int K, int rows,
                                                  const int32_t* __restrict__ root_tok,
                                                  const int32_t* __restrict__ cand_id, const float* __restrict__ U,
                                                  const float* __restrict__ Vt, int vs, float2* __restrict__ part) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* As = smem;
    unsigned char* Bs = smem + 16384;
    uint64_t* bar = (uint64_t*)(smem + 32768);
    uint32_t* tslot = (uint32_t*)(smem + 32768 + 8);
    int* fail = (int*)(smem + 32768 + 16);
    const int tid = threadIdx.x, wid = tid >> 5;
    const int split = blockIdx.x, tile = blockIdx.y;
    const int r = tile * TM + tid;
    const float NEG_INF = -__int_as_float(0x7F800000);
    const float log2e = 1.44269504088896340736f;

    if (wid == 0) dt_tmem_alloc(tslot, TN);
    if (tid == 0) {
        dt_mbar_init(bar, 1);
        dt_fence_mbar_init();
        *fail = 0;
    }
    dt_pdl_trigger();
    dt_pdl_wait();  // candidate ids and logits come from earlier kernels

    int b = 0, d = 0, u = -1;
    if (r < rows) u = row_parent(r, L, K, V, root_tok, cand_id, &b, &d);
    stage_row_bf16(As, tid, u >= 0 ? U + (size_t)u * RK : nullptr);
    const T* xrow = x + ((size_t)b * L + d) * V;
    const int vbeg = split * vs, vend = min(V, vbeg + vs);
    const uint32_t a_base = dt_smem_addr(As), b_base = dt_smem_addr(Bs);

    dt_fence_proxy_async_smem();
    dt_tc_fence_before();
    __syncthreads();
    dt_tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tlane = tmem + ((uint32_t)(wid * 32) << 16);

    float m_run = NEG_INF, s_run = 0.f;
    uint32_t phase = 0;
    // *fail is read only after a block barrier, so every thread leaves together
    for (int v0 = vbeg; v0 < vend && !*fail; v0 += TN) {
        // B tile: token v0 + tid's Vt vector (zeros past the slice)
        const int v = v0 + tid;
        stage_row_bf16(Bs, tid, v < vend ? Vt + (size_t)v * RK : nullptr);
        dt_fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            dt_tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < RK / 16; ++kk)
                dt_mma_bf16(tmem, dt_desc_kmajor_sw128(a_base + 32 * kk), dt_desc_kmajor_sw128(b_base + 32 * kk),
                            IDESC, kk > 0);
            dt_mma_commit(bar);
        }
        if (!dt_mbar_wait(bar, phase)) {
            *fail = 1;
            dt_mbar_wait(bar, phase);
        }
        phase ^= 1u;
        dt_tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < TN; c += 32) {
            float acc[32];
            dt_tmem_ld32(tlane + c, acc);
            if (u >= 0 && v0 + c < vend) {
                float xv[32];
                load_x32<T>(xrow, v0 + c, vend, xv);
                float cm = NEG_INF;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    acc[j] = __fadd_rn(acc[j], xv[j]);  // -inf past the slice
                    cm = fmaxf(cm, acc[j]);
                }
                if (cm > m_run) {
                    s_run = (m_run == NEG_INF) ? 0.f : __fmul_rn(s_run, dt_ex2_approx(__fmul_rn(__fsub_rn(m_run, cm), log2e)));
                    m_run = cm;
                }
                if (m_run != NEG_INF) {
                    float p = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) p = __fadd_rn(p, dt_ex2_approx(__fmul_rn(__fsub_rn(acc[j], m_run), log2e)));
                    s_run = __fadd_rn(s_run, p);
                }
            }
        }
        dt_tc_fence_before();
        __syncthreads();  // accumulator read and B tile consumed before the next step
    }
    __syncthreads();
    // a wait that ran out of its bound leaves the slice's sums undefined: NaN
    if (r < rows) part[(size_t)r * gridDim.x + split] = *fail ? make_float2(__int_as_float(0x7FC00000), 0.f)
                                                              : make_float2(m_run, s_run);
    if (wid == 0) {
        dt_tc_fence_after();
        dt_tmem_dealloc(tmem, TN);
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

size_t dt_kn3n_part_bytes(int rows) { return (size_t)rows * DT_KN3N_MAX_SPLIT * sizeof(float2); }

cudaError_t dt_kn3n_launch(const void* x, int dtype, int batch, int L, int K, int V, const int32_t* root_tok,
                           const int32_t* cand_id, const float* lse, const float* U, const float* Vt, float2* part,
                           float* z, cudaStream_t st) {
    const int rows = batch * L * K;
    const int mtiles = (rows + TM - 1) / TM;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms < 1) {
        (void)cudaGetLastError();
        sms = 148;
    }
    // about two CTAs per SM, vocabulary slices of whole 128-token steps
    int nsplit = (2 * sms + mtiles - 1) / mtiles;
    const int steps = (V + TN - 1) / TN;
    nsplit = max(1, min(min(nsplit, DT_KN3N_MAX_SPLIT), steps));
    const int vs = ((steps + nsplit - 1) / nsplit) * TN;
    nsplit = (V + vs - 1) / vs;
    cudaError_t e;
    DtLaunch lc(dim3(nsplit, mtiles, 1), dim3(NT, 1, 1), SMEM, st);
    if (dtype == DT_BF16) {
        if ((e = cudaFuncSetAttribute(kn3n_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) !=
            cudaSuccess)
            return e;
        e = cudaLaunchKernelEx(&lc.cfg, kn3n_kernel<uint16_t>, (const uint16_t*)x, V, L, K, rows, root_tok, cand_id, U,
                               Vt, vs, part);
    } else {
        if ((e = cudaFuncSetAttribute(kn3n_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) !=
            cudaSuccess)
            return e;
        e = cudaLaunchKernelEx(&lc.cfg, kn3n_kernel<float>, (const float*)x, V, L, K, rows, root_tok, cand_id, U, Vt,
                               vs, part);
    }
    if (e != cudaSuccess) return e;
    DtLaunch lr(dim3((rows + 255) / 256), dim3(256), 0, st);
    return cudaLaunchKernelEx(&lr.cfg, kn3n_reduce_kernel, (const float2*)part, nsplit, rows, L, K, V, root_tok,
                              cand_id, lse, z);
}
