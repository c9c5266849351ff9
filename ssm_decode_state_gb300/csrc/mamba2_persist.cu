// Launchers of the persistent Mamba-2 replay decode (float32 checkpoint; the FP16
// instantiations live in mamba2_persist_f16.cu) and of the persistent verify.
#include "mamba2_persist_launch.cuh"

namespace rssm {

rssm_status launch_decode_persistent_f16(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st);
rssm_status launch_decode_small(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st);

// Returns RSSM_ERR_UNSUPPORTED (without launching) when the shape is not one
// the persistent kernel handles; the caller then uses the per-tile kernel.
// Small batches of a float32 checkpoint without read copy take the single-pass
// kernel (mamba2_small.cu), which gives the same bits.
rssm_status launch_decode_persistent(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st) {
    if (d->ckpt_f16) return launch_decode_persistent_f16(d, args, st);
    const rssm_status s = launch_decode_small(d, args, st);
    if (s != RSSM_ERR_UNSUPPORTED) return s;
    return launch_decode_persistent_ck<0>(d, args, st);
}

// The same launch with the bounded-wait test hook on (float32 checkpoints).
rssm_status launch_decode_persistent_stalled(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st) {
    if (d->ckpt_f16) return RSSM_ERR_UNSUPPORTED;
    return launch_decode_persistent_ck<0>(d, args, st, 1);
}

}  // namespace rssm

#include "mamba2_verify_persist.cuh"

namespace rssm {

// Persistent speculative verify (serving shapes, T <= 4), then the epilogue that
// writes the drafts' B and C records.  RSSM_ERR_UNSUPPORTED (nothing launched)
// sends the caller to the per-tile kernel.
rssm_status launch_verify_persistent(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st) {
    constexpr int HPI = 8;
    if (d->ckpt_f16) return RSSM_ERR_UNSUPPORTED;     // FP16 checkpoints: the per-tile verify
    if (!d->io_bf16 || d->dstate != 128 || d->headdim != 64 || d->nheads > 4096) return RSSM_ERR_UNSUPPORTED;
    if (args.T < 1 || args.T > 4 || args.T > d->L) return RSSM_ERR_UNSUPPORTED;
    const int hpg = d->nheads / d->ngroups;
    if (hpg % HPI) return RSSM_ERR_UNSUPPORTED;
    const int sms = sm_count();
    const long long items = (long long)d->batch * d->nheads / HPI;
    if (items < 12LL * sms || items > (1LL << 30)) return RSSM_ERR_UNSUPPORTED;
    const int grid = sms;
    const int max_my = (int)((items + grid - 1) / grid);
    if (max_my > 2048) return RSSM_ERR_UNSUPPORTED;
    const int rb = 3;
    int stages = 0;
    size_t smem = 0;
    for (int s = 6; s >= 2; --s) {
        const VSmem lay(64, 128, d->L, args.T, HPI, s, rb, d->nheads, max_my);
        if (lay.total <= 227 * 1024) { stages = s; smem = lay.total; break; }
    }
    if (!stages) return RSSM_ERR_UNSUPPORTED;
    PersistCfg pc;
    pc.items = (int)items;
    pc.max_my = max_my;
    pc.nchunk = hpg / HPI;
    pc.stages = stages;
    pc.recbufs = rb;
    pc.arrivals = d->nheads / HPI;
    void *k = (void *)m2_verify_persistent<128, 64, 8, HPI>;
    rssm_status s = ensure_smem((const void *)k, smem);
    if (s != RSSM_OK) return s;
    M2Args a = args;
    void *params[] = {&a, &pc};
    if (cudaLaunchKernel(k, dim3(grid), dim3(persist_decode_threads(256)), params, smem, st) != cudaSuccess)
        return RSSM_ERR_CUDA;
    if ((s = launch_status()) != RSSM_OK) return s;
    verify_bc_epilogue<<<d->batch, 128, 0, st>>>(a);
    return launch_status();
}

}  // namespace rssm
