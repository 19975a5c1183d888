// kn5_mask.cu -- tree-attention ancestor bitmask and position ids.
//
// [DARTree] "Tree verification and DDTree": after flattening, a node may
// attend to the verified context and to the tokens on its root-to-node path;
// [DDTree] section 4.2: a token's mask follows its parent's global index.
// Row n of the mask is row parent(n) plus bit n, so rows are built level by
// level (depth 1, 2, ...) in shared memory and then streamed out coalesced.
// One CTA per request.  The arrays are validated first: root at index 0 with
// parent -1 and depth 0, every other parent in range and distinct from the
// node, depth = parent depth + 1 <= L (this also rules out cycles).
#include "dt_device.cuh"
#include "dt_launch.h"

namespace {

constexpr int NT = 512;

__global__ void __launch_bounds__(NT) kn5_kernel(int L, int Mmax, int pos_offset, const int32_t* __restrict__ parent,
                                                 const int32_t* __restrict__ depth,
                                                 const int32_t* __restrict__ n_nodes, uint32_t* __restrict__ mask,
                                                 int32_t* __restrict__ pos, int32_t* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int bad;
    __shared__ int dcount[DT_MAX_L + 2];
    __shared__ int dstart[DT_MAX_L + 2];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int Wd = (Mmax + 31) >> 5;
    int* par = (int*)smem;
    int* dep = par + Mmax;
    int* order = dep + Mmax;
    uint32_t* rows = (uint32_t*)(order + Mmax);
    dt_pdl_trigger();
    dt_pdl_wait();
    const int M = n_nodes[b];
    if (tid == 0) bad = (M < 1 || M > Mmax) ? 1 : 0;
    if (tid < DT_MAX_L + 2) dcount[tid] = 0;
    __syncthreads();
    if (bad) {
        if (tid == 0) atomicOr(&status[b], DT_DEV_BAD_TREE);
        return;
    }
    const size_t tb = (size_t)b * Mmax;
    for (int n = tid; n < M; n += NT) {
        par[n] = parent[tb + n];
        dep[n] = depth[tb + n];
    }
    __syncthreads();
    for (int n = tid; n < M; n += NT) {
        const int p = par[n], d = dep[n];
        bool ok;
        if (n == 0) ok = (p == -1 && d == 0);
        else ok = (p >= 0 && p < M && p != n && d >= 1 && d <= L && d == dep[p] + 1);
        if (!ok) bad = 1;
        else atomicAdd(&dcount[d], 1);
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) atomicOr(&status[b], DT_DEV_BAD_TREE);
        return;
    }
    if (tid == 0) {
        int a = 0;
        for (int d = 0; d <= L; ++d) { dstart[d] = a; a += dcount[d]; dcount[d] = 0; }
        dstart[L + 1] = a;
    }
    __syncthreads();
    for (int n = tid; n < M; n += NT) {
        const int d = dep[n];
        order[dstart[d] + atomicAdd(&dcount[d], 1)] = n;
    }
    // row of the root: bit 0 only
    for (int w = tid; w < Wd; w += NT) rows[w] = (w == 0) ? 1u : 0u;
    __syncthreads();
    for (int d = 1; d <= L; ++d) {
        const int s0 = dstart[d], cnt = dstart[d + 1] - s0;
        if (cnt == 0) break;
        for (int t = tid; t < cnt * Wd; t += NT) {
            const int n = order[s0 + t / Wd];
            const int w = t % Wd;
            uint32_t v = rows[(size_t)par[n] * Wd + w];
            if (w == (n >> 5)) v |= 1u << (n & 31);
            rows[(size_t)n * Wd + w] = v;
        }
        __syncthreads();
    }
    uint32_t* out = mask + tb * Wd;
    for (int i = tid; i < M * Wd; i += NT) out[i] = rows[i];
    for (int n = tid; n < M; n += NT) pos[tb + n] = dep[n] + pos_offset;
}

}  // namespace

size_t dt_kn5_smem_bytes(int Mmax) {
    const int Wd = (Mmax + 31) >> 5;
    return (size_t)Mmax * 12 + (size_t)Mmax * Wd * 4;
}

cudaError_t dt_kn5_launch(int batch, int L, int Mmax, int pos_offset, const int32_t* parent, const int32_t* depth,
                          const int32_t* n_nodes, uint32_t* mask, int32_t* pos, int32_t* status, cudaStream_t st) {
    const size_t smem = dt_kn5_smem_bytes(Mmax);
    cudaError_t e = cudaFuncSetAttribute(kn5_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    DtLaunch lc(dim3(batch), dim3(NT), smem, st);
    return cudaLaunchKernelEx(&lc.cfg, kn5_kernel, L, Mmax, pos_offset, parent, depth, n_nodes, mask, pos, status);
}
