// Launcher of the persistent Mamba-2 replay decode (serving shapes), shared by the
// translation units that instantiate it for a float32 and for an FP16 checkpoint.
#pragma once

#include <algorithm>

#include "host_common.h"
#include "mamba2_persist.cuh"

namespace rssm {

// float4s per consumer thread per head tile: 8 -> 8 consumer warps of 8 rows each
constexpr int kPersistVPT = 8;

// Returns RSSM_ERR_UNSUPPORTED (without launching) when the shape is not one
// the persistent kernel handles; the caller then uses the per-tile kernel.
// CK: checkpoint precision of the instantiations (0 float32, 1 FP16).
// stall = 1 is the bounded-wait test hook (the consumers' first wait runs out).
template <int CK>
rssm_status launch_decode_persistent_ck(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st,
                                        int stall = 0) {
    if (!d->io_bf16 || d->dstate != 128 || d->headdim != 64 || d->nheads > 4096) return RSSM_ERR_UNSUPPORTED;
    const int hpg = d->nheads / d->ngroups;
    const int sms = sm_count();
    // heads per work item: the largest item that still leaves about one item per SM
    // (items >= 4/5 of the SMs).  An item's preparation (records, weights, record
    // term) is a chain of dependent latencies, so fewer, larger items win as long as
    // the SMs stay busy; measured at batches 1-192 (us per step with 1 / 2 / 4 / 8
    // heads per item): batch 2 8.97 / 7.85 / 8.66 / 11.18, batch 8 18.19 / 13.78 /
    // 11.61 / 11.37, batch 64 112.4 / 65.6 / 49.1 / 48.7, batch 192 329.8 / 181.8 /
    // 140.4 / 134.0
    int hpi = 1;
    for (int c : {8, 4, 2, 1}) {
        if (hpg % c) continue;
        if ((long long)d->batch * d->nheads / c * 5 >= 4LL * sms) { hpi = c; break; }
    }
    const long long items = (long long)d->batch * d->nheads / hpi;
    // every batch: at batches 1-2 (fewer items than SMs) the persistent kernel still
    // beats the per-tile kernel (7.3 vs 15.0 us at batch 1, 7.9 vs 12.1 at batch 2)
    if (items < 1 || items > (1LL << 30)) return RSSM_ERR_UNSUPPORTED;
    const int grid = (int)(items < sms ? items : sms);
    const int max_my = (int)((items + grid - 1) / grid);   // ring pointers of these are kept in smem
    if (max_my > 2048) return RSSM_ERR_UNSUPPORTED;
    int stages = 0, recbufs = 0;
    size_t smem = 0;
    for (int s = 6; s >= 2; --s) {
        // record buffers: records of item k+1 land while item k is consumed, and the
        // next item's preparation reads them during item k
        const int rb = std::min(8, std::max(3, (s + hpi - 1) / hpi + 2));
        const PSmem lay(64, 128, d->L, hpi, s, rb, d->nheads, max_my, d->read_copy, CK);
        if (lay.total <= 227 * 1024) { stages = s; recbufs = rb; smem = lay.total; break; }
    }
    if (!stages) return RSSM_ERR_UNSUPPORTED;
    PersistCfg pc;
    pc.items = (int)items;
    pc.max_my = max_my;
    pc.nchunk = hpg / hpi;
    pc.stages = stages;
    pc.recbufs = recbufs;
    pc.arrivals = d->nheads / hpi;
    pc.stall = stall;
    constexpr int VPT = kPersistVPT;
    void *k = nullptr;
#define RSSM_PD(RC)                                                                         \
    switch (hpi) {                                                                          \
        case 8: k = (void *)m2_decode_persistent<128, 64, VPT, 8, RC, CK>; break;              \
        case 4: k = (void *)m2_decode_persistent<128, 64, VPT, 4, RC, CK>; break;              \
        case 2: k = (void *)m2_decode_persistent<128, 64, VPT, 2, RC, CK>; break;              \
        default: k = (void *)m2_decode_persistent<128, 64, VPT, 1, RC, CK>; break;             \
    }
    if (d->read_copy == 2) { RSSM_PD(2) }
    else if (d->read_copy == 1) { RSSM_PD(1) }
    else { RSSM_PD(0) }
#undef RSSM_PD
    rssm_status s = ensure_smem((const void *)k, smem);
    if (s != RSSM_OK) return s;
    M2Args a = args;
    void *params[] = {&a, &pc};
    const int threads = persist_decode_threads(64 * 128 / 4 / VPT);
    if (cudaLaunchKernel(k, dim3(grid), dim3(threads), params, smem, st) != cudaSuccess) return RSSM_ERR_CUDA;
    return launch_status();
}

}  // namespace rssm
