// kn0_ceiling.cu -- the read floor of the few-row stage-1 launch.
//
// A measurement kernel, not a step of the method: it reads the drafter rows
// with exactly the launch that the cluster stage-1 kernel (kn1_candidates.cu)
// gets -- the same grid of S-CTA clusters, one per row, the same chunk per
// CTA, the same residency (one CTA per SM), programmatic dependent launch --
// and does the least work that still consumes every
// byte: each CTA bulk-copies its chunk into shared memory, takes the chunk's
// maximum in one pass and writes it.  No exchange between the CTAs.  Its
// device time bounds from below what any kernel of that launch shape can
// reach on the same bytes; the stage-1 kernel's time over it shows what its
// own exchanges and passes cost.
#include "dt_launch.h"
#include "kn1_common.cuh"

namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr size_t kOneCtaSmem = 120 * 1024;  // above half of an SM's shared memory

template <typename T>
__global__ void __launch_bounds__(NT, 1) kn0_kernel(const T* __restrict__ logits, int V, int chunk, int S,
                                                     size_t data_off, float* __restrict__ out,
                                                     int32_t* __restrict__ timed_out) {
    constexpr int EPV = 16 / sizeof(T);
    const float NEG_INF = -__int_as_float(0x7F800000);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bar;
    __shared__ float red[NW];
    const int c = blockIdx.x, row = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int lo = min(V, c * chunk), hi = min(V, lo + chunk);
    unsigned char* data = smem + data_off;

    if (tid == 0) {
        dt_mbar_init(&bar, 1);
        dt_fence_mbar_init();
    }
    dt_pdl_trigger();
    __syncthreads();
    dt_pdl_wait();
    DtStager<T> stg;
    const bool pend = stg.start(logits + (size_t)row * (size_t)V, lo, hi, data, &bar) != 0;
    stg.finish(data);
    if (pend && tid == 0 && !dt_mbar_wait(&bar, 0)) {
        if (timed_out) atomicOr(timed_out, DT_DEV_TIMEOUT);
        dt_mbar_wait(&bar, 0);  // the copy must land before the CTA may exit
    }
    __syncthreads();

    const int h = (int)(((uintptr_t)(logits + (size_t)row * (size_t)V + lo) & 15u) / sizeof(T));
    const int n = hi - lo;
    const int nv = (h + n + EPV - 1) / EPV;
    const int full_lo = h > 0 ? 1 : 0;
    const int full_hi = ((h + n) % EPV == 0) ? nv : nv - 1;
    const uint4* v = (const uint4*)data;
    float m = NEG_INF;
    for (int j = tid; j < nv; j += NT) {
        const uint4 q = v[j];
        if (j >= full_lo && j < full_hi) {
            m = fmaxf(m, dt_vec_max<T>(q));
        } else {
            float x[EPV];
            dt_vec_vals<T>(q, x);
#pragma unroll
            for (int s = 0; s < EPV; ++s) {
                const int idx = j * EPV + s - h;
                if (idx >= 0 && idx < n) m = fmaxf(m, x[s]);
            }
        }
    }
    m = dt_warp_max(m);
    if (lane == 0) red[wid] = m;
    __syncthreads();
    if (tid == 0) {
        float a = NEG_INF;
#pragma unroll
        for (int w = 0; w < NW; ++w) a = fmaxf(a, red[w]);
        out[(size_t)row * S + c] = a;
    }
}

}  // namespace

cudaError_t dt_kn0_launch(const void* logits, int dtype, int rows, int V, int Kc, int S, int chunk, float* out,
                          int32_t* timed_out, cudaStream_t st) {
    const int esize = dtype == DT_BF16 ? 2 : 4;
    // the stage-1 kernel's dynamic shared memory (its data area sits at the
    // end), and at least half an SM's, so that -- like the stage-1 kernel,
    // whose registers allow one CTA per SM -- no two CTAs share an SM
    const size_t need = dt_kn1_smem_bytes(chunk, Kc, esize);
    const size_t smem = need > kOneCtaSmem ? need : kOneCtaSmem;
    const size_t data_off = need - (size_t)chunk * esize - 32;
    DtLaunch lc(dim3(S, rows, 1), dim3(NT, 1, 1), smem, st, S);
    cudaError_t e;
    if (dtype == DT_BF16) {
        e = cudaFuncSetAttribute(kn0_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess && S > 8)
            e = cudaFuncSetAttribute(kn0_kernel<uint16_t>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&lc.cfg, kn0_kernel<uint16_t>, (const uint16_t*)logits, V, chunk, S, data_off, out,
                                  timed_out);
    }
    e = cudaFuncSetAttribute(kn0_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && S > 8)
        e = cudaFuncSetAttribute(kn0_kernel<float>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&lc.cfg, kn0_kernel<float>, (const float*)logits, V, chunk, S, data_off, out, timed_out);
}
