// Helpers shared by the persistent (one CTA per SM, warp-specialised) kernels.
#pragma once

#include "common.cuh"

namespace rssm {

// Threads of the item-preparation warps of the persistent decode kernels.
constexpr int kPrepThreads = 64;

__device__ __forceinline__ float bf16_at(const uint16_t *p, int i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}

// cp.async completion of this thread's earlier copies counts as one arrival
// on `bar` (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Named barrier among the NC consumer threads only.
template <int NC>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
}

// Named barrier among the item-preparation warps only.
__device__ __forceinline__ void prep_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kPrepThreads) : "memory"); }

// Packed pair of float32 (one 64-bit register) and the sm_100+ two-wide fma:
// each lane of the pair is an ordinary fused multiply-add, rounded once.
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Bounded wait that also gives up as soon as another warp has aborted.
__device__ __forceinline__ bool pwait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    // The clock is read only once a wait has polled 256 times: reading it is
    // slow, and short waits sit on the path that hands a stage to the consumers.
    uint64_t t0 = 0;
    for (uint32_t it = 1; it <= (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort_flag) return false;
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > 2000000000ull) return false;
        }
    }
    return false;
}

}  // namespace rssm
