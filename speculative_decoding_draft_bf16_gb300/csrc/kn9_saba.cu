// kn9_saba.cu -- SABA: state-aware per-request tree budgets.
//
// [GRAFT] "State-aware budget allocation": per decoding round t the state
// s_t = [conf, degen, hist] (conf: mean over the block positions of the
// drafter's top-candidate probability; degen: mean cosine similarity of
// adjacent drafter hidden states plus its growth r_{D-1} - r_1; hist: mean
// accepted length over the last w rounds), the gain G(B) = a * B^0.5 with
// a = mean of (l + 1) over the same rounds, the cost C(B) = B * c_verify +
// c_fixed, and B_t = argmax_B G(B) / C(B) over the integers [B_min, B_max]
// (smallest B on ties).  As printed, a cancels in the argmax (the optimum is
// c_fixed / c_verify); the state is still computed and reported.
//
// One CTA per request: one thread updates the history ring with the last
// round's accepted length and forms hist and a; the warps take the
// adjacent-position cosines; every thread scores a share of the budgets with
// (a * sqrt(B)) / (B * c_verify + c_fixed), one rounding per operation, and a
// block max over (score, -B) keys picks the budget.
#include "dt_device.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT9 = 256;
constexpr int NW9 = NT9 / 32;

__global__ void __launch_bounds__(NT9) kn9_kernel(int L, int Kc, const float* __restrict__ cand_lp,
                                                  const float* __restrict__ hidden, int Hd,
                                                  const int32_t* __restrict__ prev_len, int32_t* __restrict__ ring,
                                                  int32_t* __restrict__ count, int w, float c_verify, float c_fixed,
                                                  int B_min, int B_max, float* __restrict__ state,
                                                  int32_t* __restrict__ budget) {
    __shared__ float sh_a, sh_hist, sh_conf;
    __shared__ float sh_r[DT_MAX_L];
    __shared__ unsigned long long sh_best[NW9];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    dt_pdl_trigger();
    dt_pdl_wait();  // candidate tables and accepted lengths come from earlier kernels
    if (tid == 0) {
        int32_t* rb = ring + (size_t)b * w;
        int cnt = count[b];
        if (prev_len && prev_len[b] >= 0) {
            rb[cnt % w] = prev_len[b];
            ++cnt;
            count[b] = cnt;
        }
        const int n = cnt < w ? cnt : w;
        long long sum = 0;
        for (int i = 0; i < n; ++i) sum += rb[(cnt - 1 - i) % w];
        sh_hist = n ? __fdiv_rn((float)sum, (float)n) : 0.f;
        sh_a = n ? __fdiv_rn((float)(sum + n), (float)n) : 1.f;
        float c = 0.f;
        for (int d = 0; d < L; ++d) c += expf(cand_lp[((size_t)b * L + d) * Kc]);
        sh_conf = c / (float)L;
    }
    // adjacent-position cosines of the drafter hidden states, one warp per pair
    if (hidden) {
        const float* h = hidden + (size_t)b * L * Hd;
        for (int d = wid; d + 1 < L; d += NW9) {
            float dot = 0.f, n1 = 0.f, n2 = 0.f;
            for (int k = lane; k < Hd; k += 32) {
                const float x = h[(size_t)d * Hd + k], y = h[(size_t)(d + 1) * Hd + k];
                dot = fmaf(x, y, dot);
                n1 = fmaf(x, x, n1);
                n2 = fmaf(y, y, n2);
            }
            dot = dt_warp_sum(dot);
            n1 = dt_warp_sum(n1);
            n2 = dt_warp_sum(n2);
            if (lane == 0) sh_r[d] = (n1 > 0.f && n2 > 0.f) ? dot / sqrtf(n1 * n2) : 0.f;
        }
    }
    __syncthreads();
    // budget: the best (score, smallest B)
    const float a = sh_a;
    unsigned long long best = 0;
    for (int B = B_min + tid; B <= B_max; B += NT9) {
        const float fb = (float)B;
        const float u = __fdiv_rn(__fmul_rn(a, __fsqrt_rn(fb)), __fadd_rn(__fmul_rn(fb, c_verify), c_fixed));
        const unsigned long long key =
            ((unsigned long long)__float_as_uint(u) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)B);
        best = key > best ? key : best;  // u > 0: its bit pattern orders like the value
    }
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
        best = t > best ? t : best;
    }
    if (lane == 0) sh_best[wid] = best;
    __syncthreads();
    if (tid == 0) {
        unsigned long long g = 0;
        for (int i = 0; i < NW9; ++i) g = sh_best[i] > g ? sh_best[i] : g;
        budget[b] = (int32_t)(0xFFFFFFFFu - (uint32_t)(g & 0xFFFFFFFFull));
        float degen = 0.f;
        if (hidden && L >= 2) {
            float rs = 0.f;
            for (int d = 0; d + 1 < L; ++d) rs += sh_r[d];
            degen = rs / (float)(L - 1) + (sh_r[L - 2] - sh_r[0]);
        }
        float* st = state + (size_t)b * 4;
        st[0] = sh_conf;
        st[1] = degen;
        st[2] = sh_hist;
        st[3] = a;
    }
}

}  // namespace

cudaError_t dt_kn9_launch(int batch, int L, int Kc, const float* cand_lp, const float* hidden, int Hd,
                          const int32_t* prev_len, int32_t* ring, int32_t* count, int w, float c_verify,
                          float c_fixed, int B_min, int B_max, float* state, int32_t* budget, cudaStream_t st) {
    DtLaunch lc(dim3(batch), dim3(NT9), 0, st);
    return cudaLaunchKernelEx(&lc.cfg, kn9_kernel, L, Kc, cand_lp, hidden, Hd, prev_len, ring, count, w, c_verify,
                              c_fixed, B_min, B_max, state, budget);
}
