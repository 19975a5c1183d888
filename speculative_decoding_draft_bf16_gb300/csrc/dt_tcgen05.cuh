// dt_tcgen05.cuh -- fifth-generation tensor core (tcgen05) helpers, sm_100a+.
//
// Tensor memory (TMEM) holds the accumulators: 128 lanes x 512 32-bit columns
// per SM, allocated in power-of-two column blocks by one warp.  An MMA is
// issued by a single thread; its operands are read from shared memory through
// 64-bit matrix descriptors; completion is signalled on an mbarrier with
// tcgen05.commit; the accumulator is read back to registers with tcgen05.ld.
#pragma once

#include "dt_device.cuh"

// ---- TMEM allocation (one full warp) ---------------------------------------
// Allocates ncols columns (power of two, >= 32) and writes the TMEM address to
// the shared-memory word `dst`.
DT_DI void dt_tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dt_smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
DT_DI void dt_tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations around thread synchronisation.
DT_DI void dt_tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DT_DI void dt_tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads).
DT_DI void dt_fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- shared-memory matrix descriptor -----------------------------------------
// K-major operand tile with 128-byte swizzling: rows of 128 bytes (64 bf16),
// 8-row atoms of 1 KB stacked along M (or N); the tile base is 1024-byte
// aligned.  Row r's 16-byte chunk c is stored at chunk c ^ (r % 8).
// Fields: start address >> 4 (bits 0-13), leading-dimension byte offset >> 4
// (16-29; unused within one 128-byte swizzle span, set to 1), stride byte
// offset >> 4 (32-45: 1024 B between 8-row atoms), descriptor version 1
// (bits 46-47), base offset 0, swizzle mode 2 = 128 B (bits 61-63).
DT_DI uint64_t dt_desc_kmajor_sw128(uint32_t smem_addr) {
    return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Byte offset of element (row r, k) (16-bit elements, k < 64) in such a tile.
DT_DI uint32_t dt_sw128_offset(int r, int k) {
    const uint32_t b = (uint32_t)k * 2u;
    return (uint32_t)r * 128u + ((((b >> 4) ^ (uint32_t)(r & 7)) << 4) | (b & 15u));
}

// ---- instruction descriptor, kind::f16 ---------------------------------------
// bf16 A and B (both K-major), fp32 accumulator, shape M x N:
// D format f32 (bits 4-5 = 1), A format bf16 (7-9 = 1), B format bf16
// (10-12 = 1), no negation, K-major A and B (bits 15, 16 = 0), N >> 3
// (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t dt_idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A * B^T for one K step of 16, issued by one thread.
DT_DI void dt_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// Arrives on the mbarrier once every tcgen05 operation issued so far by this
// thread has completed.
DT_DI void dt_mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     dt_smem_addr(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w of a
// warpgroup reads lanes 32*(w%4) .. +31; taddr includes that lane offset).
// The load and its completion wait are one asm statement, so no use of the
// registers can be scheduled before the data has arrived.
DT_DI void dt_tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
