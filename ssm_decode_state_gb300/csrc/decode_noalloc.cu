// replayssm_decode_noalloc: the replay decode for callers that cannot
// allocate device memory.
//
// The replay decode kernels need one piece of scratch memory besides the
// caller's cache: a per-sequence arrival counter (cache->arrive), which the
// CTAs of a sequence count up on so that the last one can commit the ring
// pointers.  Some callers have no way to provide it: a plugin inside an
// inference engine whose memory planner owns all device memory and hands the
// plugin only its inputs and outputs, or code that holds no device buffer of
// its own from one call to the next.  This entry point keeps those counters
// in a fixed array in the library's own device memory instead, so it never
// allocates.
#include <mutex>

#include "host_common.h"

namespace {

constexpr int kNoAllocMaxBatch = 4096;   // sequences per call; 16 KiB of counters

// Arrival counters shared by every call on a device.  Each GPU that loads the
// library keeps this array until the process exits.  In host code the name
// is only a stand-in for the symbol, never a device address.
static __device__ __align__(256) int32_t g_arrive_scratch[kNoAllocMaxBatch];

std::mutex g_setup_mutex;
int32_t *g_scratch_ptr[64] = {nullptr};

// Device address of the counters on the current device, looked up once per
// device (with that device current) and kept for the life of the process: a
// cudaDeviceReset reloads the library's device code elsewhere, so the cached
// address would then be stale (the header forbids use across a reset).
rssm_status scratch_for_current_device(int32_t **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RSSM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_arrive_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return RSSM_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_scratch_ptr[dev];
    return RSSM_OK;
}

}  // namespace

extern "C" rssm_status replayssm_decode_noalloc(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                                                const float *dt, const void *x, const void *B, const void *C,
                                                float *y, void *stream) {
    // every host-side check first, so that a call rejected here enqueues nothing
    // (in particular, clears no counters another call may still be using)
    rssm::TileGeom geom;
    rssm_status v = rssm::check_decode_call(dims, cache, dt, x, B, C, y, false, &geom);
    if (v != RSSM_OK) return v;
    // the counters are indexed by cache slot: the cache's capacity (batch without a
    // slot map) must fit the fixed array
    const int cap = cache->capacity > 0 ? cache->capacity : dims->batch;
    if (cap > kNoAllocMaxBatch) return RSSM_ERR_SHAPE;
    int32_t *scratch = nullptr;
    rssm_status s = scratch_for_current_device(&scratch);
    if (s != RSSM_OK) return s;
    // the counters must start at zero; a call that was abandoned could have
    // left some behind, so clear this call's share first (stream-ordered)
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, sizeof(int32_t) * (size_t)cap, st) != cudaSuccess) {
        cudaGetLastError();
        return RSSM_ERR_CUDA;
    }
    rssm_mamba2_cache c = *cache;
    c.arrive = scratch;
    return replayssm_decode(dims, &c, dt, x, B, C, y, stream);
}
