// dt_mask.cuh -- the tree-attention mask rows that the selection kernels
// write beside their trees (the fused select + mask path).
#pragma once

#include "dt_device.cuh"

// Tree-attention mask rows of one request's tree, written by the CTA that
// holds the tree in shared memory: bit m % 32 of word m / 32 of row n is set
// iff node m is n or one of its ancestors.  parent_of(n) gives node n's parent
// index (-1 for the root, node 0) from shared memory, so walking a chain costs
// shared-memory latency only.  The M rows are zeroed first with coalesced
// stores; after a barrier each thread walks its rows' chains.  Parents precede
// their children in every tree the selection kernels write, so a chain visits
// words in non-increasing order and each nonzero word is stored once; a
// parent index that does not precede its child (a tree built from non-finite
// scores, which the status reports) ends the chain there, so that no index
// outside the tree is ever followed.  Block-uniform; contains one
// __syncthreads.
template <int NT, typename ParentOf>
DT_DI void dt_write_mask_rows(int M, int Mmax, ParentOf parent_of, uint32_t* mask) {
    const int Wd = (Mmax + 31) >> 5;
    for (int i = threadIdx.x; i < M * Wd; i += NT) mask[i] = 0u;
    __syncthreads();
    for (int n = threadIdx.x; n < M; n += NT) {
        uint32_t* row = mask + (size_t)n * Wd;
        int w = n >> 5;
        uint32_t bits = 1u << (n & 31);
        for (int prev = n, a = parent_of(n); a >= 0 && a < prev; prev = a, a = parent_of(a)) {
            if ((a >> 5) != w) {
                row[w] = bits;
                w = a >> 5;
                bits = 0u;
            }
            bits |= 1u << (a & 31);
        }
        row[w] = bits;
    }
}
