// Fifth-generation tensor core (tcgen05) helpers for sm_100a / sm_103a:
// tensor-memory allocation, shared-memory matrix descriptors, the bf16 MMA with
// a float32 accumulator in tensor memory, its completion signal, and the
// tensor-memory to register load.  Inline PTX only.
//
// Every operand these kernels hand to the tensor core is K-major with the
// 128-byte swizzle: a K-block of 64 bf16 per row (128 bytes), rows in groups of
// eight (1024 bytes, the swizzle atom), groups one after another; inside a row
// the 16-byte chunk c of row r sits at chunk position c ^ (r mod 8).  An MMA
// of K = 16 reads 32 bytes of every row, so successive K steps inside a
// K-block start 32 bytes further on.  Atoms must start on 1024-byte
// boundaries.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace rssm {
namespace tc {

// Byte offset of element (row, k) of a K-major, 128-byte-swizzled K-block of
// bf16 (k < 64).
__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int k) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 3) ^ row) & 7) << 4) + (k & 7) * 2);
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// whose first row starts at shared address saddr: stride between 8-row groups
// 1024 bytes (the leading-dimension offset is unused by this layout).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and a
// float32 accumulator, for an M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Tensor-memory allocation of ncols columns (a power of two >= 32) by one
// whole warp; the base address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tensor-core operations around thread synchronisation.
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Makes this thread's shared-memory stores visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, one thread issues; acc = false starts D afresh.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}

// One arrival on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Warp-wide load of 32 tensor-memory lanes x 32 columns of 32 bits starting at
// taddr (lane in the upper 16 bits, column in the lower): thread t receives
// lane (taddr >> 16) + t, columns c .. c + 31.  The wait is in the same asm
// statement, so the registers are complete when it returns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
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

// Two floats to a bf16 pair, round to nearest even: lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// x = t1 + t2 + t3 exactly for float32 x = 0 or 2^-110 <= |x| <= the largest
// finite bf16 (~3.39e38): t1 the nearest bf16 to x, t2 the nearest to x - t1
// (exact in float32), t3 = x - t1 - t2 (at most eight significant bits are left,
// so it is a bf16 itself).  Below that range t3 would be subnormal and lose bits;
// above it t1 rounds to infinity.  Two values per call, as bf16 pairs.
__device__ __forceinline__ void split3_bf16x2(float x0, float x1, uint32_t &t1, uint32_t &t2, uint32_t &t3) {
    t1 = bf16x2_rn(x0, x1);
    float r0 = x0 - __uint_as_float(t1 << 16), r1 = x1 - __uint_as_float(t1 & 0xffff0000u);
    t2 = bf16x2_rn(r0, r1);
    r0 -= __uint_as_float(t2 << 16);
    r1 -= __uint_as_float(t2 & 0xffff0000u);
    t3 = bf16x2_rn(r0, r1);
}

}  // namespace tc
}  // namespace rssm
