// Host-side helpers shared by the entry points: argument checks, launch
// geometry, error mapping.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "replayssm.h"

namespace rssm {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

inline rssm_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

// Allow a kernel more than 48 KiB of dynamic shared memory when it needs it.
template <typename K>
inline rssm_status ensure_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return RSSM_OK;
    if (bytes > 227 * 1024) return RSSM_ERR_SHAPE;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return RSSM_ERR_CUDA;
    return RSSM_OK;
}

// Launch geometry of a (sequence, head) checkpoint tile of `rows` x `cols`
// floats split `split` ways along the rows: R rows per CTA, VPT float4 per
// thread, `threads` per CTA.  The tile rows of a CTA start on a multiple of 8
// (16-byte record chunks) and every warp is full.
struct TileGeom {
    int split, R, vpt, threads;
};

inline bool tile_geom_ok(int R, int cols, int vpt, int max_threads) {
    const int f4 = R * cols / 4;
    if (R % 8 != 0 || f4 % vpt != 0) return false;
    const int t = f4 / vpt;
    return t >= 32 && t % 32 == 0 && t <= max_threads;
}

// Choose the smallest split that fits and then split further while the grid
// has fewer than ~4 CTAs per SM (small batches), as long as the tile stays a
// valid shape.
inline bool choose_geom(int batch, int heads, int rows, int cols, TileGeom &g, int max_threads = 256) {
    const int target = 4 * sm_count();
    g.split = 0;
    for (int s = 1; s <= rows / 8; s *= 2) {
        if (rows % s) break;
        const int R = rows / s;
        int vpt = 0;
        if (tile_geom_ok(R, cols, 8, max_threads)) vpt = 8;
        else if (tile_geom_ok(R, cols, 2, max_threads)) vpt = 2;
        if (!vpt) {
            if (g.split) break;   // cannot split further
            continue;             // tile still too large: try a finer split
        }
        g.split = s; g.R = R; g.vpt = vpt; g.threads = R * cols / 4 / vpt;
        if ((long long)batch * heads * s >= target) break;
    }
    return g.split > 0;
}

// All host-side checks of a replay decode call (dims, cache, token buffers,
// launch geometry); need_arrive = false accepts a cache without arrival counters.
rssm_status check_decode_call(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c, const float *dt,
                              const void *x, const void *B, const void *C, const float *y, bool need_arrive,
                              TileGeom *geom);

// Device-side ring rollback shared by the Mamba-2 and GDN caches (launch only).
rssm_status launch_ring_rollback(int batch, int L, int T, const int32_t *accepted, const int32_t *slots, int cap,
                                 int32_t *ring_head, int32_t *ring_len, uint32_t *err, cudaStream_t st);

}  // namespace rssm
