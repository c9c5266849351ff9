// Entry points of the Mamba-2 replay path: decode, standalone flush, verify,
// rollback and the read-copy rebuild.
#include "host_common.h"
#include "mamba2_replay.cuh"

namespace rssm {

rssm_status launch_decode_persistent(const rssm_mamba2_dims *d, const M2Args &a, cudaStream_t st);
rssm_status launch_verify_persistent(const rssm_mamba2_dims *d, const M2Args &a, cudaStream_t st);
rssm_status launch_decode_persistent_stalled(const rssm_mamba2_dims *d, const M2Args &a, cudaStream_t st);

namespace {

rssm_status check_dims(const rssm_mamba2_dims *d) {
    if (!d) return RSSM_ERR_NULL;
    if (d->batch < 1 || d->nheads < 1 || d->ngroups < 1 || d->nheads % d->ngroups) return RSSM_ERR_SHAPE;
    if (!(d->dstate == 16 || d->dstate == 32 || d->dstate == 64 || d->dstate == 128)) return RSSM_ERR_SHAPE;
    if (d->headdim < 8 || d->headdim > 256 || d->headdim % 8) return RSSM_ERR_SHAPE;
    if (d->L < 1 || d->L > kMaxL) return RSSM_ERR_SHAPE;
    if (d->read_copy < 0 || d->read_copy > 2) return RSSM_ERR_SHAPE;   // none, FP8 E4M3, NVFP4
    if (d->io_bf16 != 0 && d->io_bf16 != 1) return RSSM_ERR_SHAPE;
    if (d->ckpt_f16 != 0 && d->ckpt_f16 != 1) return RSSM_ERR_SHAPE;
    if (d->batch > 65535) return RSSM_ERR_SHAPE;
    return RSSM_OK;
}

rssm_status check_cache(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c) {
    if (!c) return RSSM_ERR_NULL;
    if (!c->ckpt || !c->rec_dt || !c->rec_x || !c->rec_B || !c->ring_head || !c->ring_len ||
        !c->arrive || !c->A || !c->D || !c->err)
        return RSSM_ERR_NULL;
    if (d->read_copy && (!c->ckpt_q || !c->ckpt_scale)) return RSSM_ERR_NULL;
    if (!aligned16(c->ckpt) || !aligned16(c->rec_x) || !aligned16(c->rec_B) ||
        (c->rec_C && !aligned16(c->rec_C)) || (d->read_copy && (!aligned16(c->ckpt_q) || !aligned16(c->ckpt_scale))))
        return RSSM_ERR_ALIGN;
    if (c->capacity < 0 || (!c->slots && c->capacity > 0 && c->capacity < d->batch)) return RSSM_ERR_SHAPE;
    return RSSM_OK;
}

int cache_capacity(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c) {
    return c->capacity > 0 ? c->capacity : d->batch;
}

template <int MODE, int TQ>
void *pick_kernel(int N, int vpt) {
#define RSSM_PICK(NN)                                                                  \
    if (N == NN) return vpt == 8 ? (void *)m2_replay_kernel<MODE, NN, 8, TQ>           \
                                 : (void *)m2_replay_kernel<MODE, NN, 2, TQ>;
    RSSM_PICK(16) RSSM_PICK(32) RSSM_PICK(64) RSSM_PICK(128)
#undef RSSM_PICK
    return nullptr;
}

M2Args make_args(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c, const TileGeom &g) {
    M2Args a{};
    a.B = d->batch; a.H = d->nheads; a.P = d->headdim; a.N = d->dstate; a.G = d->ngroups;
    a.L = d->L; a.R = g.R; a.split = g.split; a.T = 0; a.hpg = d->nheads / d->ngroups;
    a.read_copy = d->read_copy; a.io_bf16 = d->io_bf16;
    a.ckpt = static_cast<float *>(c->ckpt); a.ckpt_q = c->ckpt_q; a.ckpt_scale = c->ckpt_scale;
    a.ckpt_f16 = d->ckpt_f16;
    a.seed_lo = (uint32_t)(c->sr_seed & 0xffffffffu); a.seed_hi = (uint32_t)(c->sr_seed >> 32);
    a.rec_dt = c->rec_dt; a.rec_x = c->rec_x; a.rec_B = c->rec_B; a.rec_C = c->rec_C;
    a.ring_head = c->ring_head; a.ring_len = c->ring_len; a.arrive = c->arrive;
    a.A = c->A; a.D = c->D; a.err = c->err;
    a.slots = c->slots; a.cap = cache_capacity(d, c);
    return a;
}

template <int MODE, int TQ>
rssm_status launch(const rssm_mamba2_dims *d, M2Args &a, const TileGeom &g, cudaStream_t st) {
    void *k = pick_kernel<MODE, TQ>(d->dstate, g.vpt);
    if (!k) return RSSM_ERR_UNSUPPORTED;
    const M2Smem lay(MODE, d->L, MODE == kVerify ? a.T : 0, g.R, d->dstate);
    const size_t smem = (size_t)lay.total * sizeof(float);
    rssm_status s = ensure_smem((const void *)k, smem);
    if (s != RSSM_OK) return s;
    void *params[] = {&a};
    if (cudaLaunchKernel(k, dim3(d->nheads * g.split, d->batch), dim3(g.threads), params, smem, st) !=
        cudaSuccess)
        return RSSM_ERR_CUDA;
    return launch_status();
}

__global__ void rollback_kernel(int batch, int L, int T, const int32_t *accepted, const int32_t *slots, int cap,
                                int32_t *ring_head, int32_t *ring_len, uint32_t *err) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int sb = slots ? slots[b] : b;
    if (sb < 0 || sb >= cap) {
        flag_error(err, RSSM_DEVERR_SLOT);
        return;
    }
    const int head = ring_head[sb], len = ring_len[sb], acc = accepted[b];
    if (head < 0 || head >= L || len < 0 || len > L) {
        flag_error(err, RSSM_DEVERR_RING_META);
        return;
    }
    if (acc < 0 || acc > T || len < T - acc) {
        flag_error(err, RSSM_DEVERR_ROLLBACK);
        return;
    }
    ring_len[sb] = len - (T - acc);
}

// One thread per float4 of the checkpoint; the N/4 lanes of a row agree on
// its maximum with shuffles.
// Four consecutive checkpoint values (float32, or FP16 when f16).
__device__ __forceinline__ float4 ckpt_load4(const void *ckpt, long long i, int f16) {
    return f16 ? f16x4_to_float4(__ldcs(reinterpret_cast<const uint2 *>(ckpt) + i))
               : __ldcs(reinterpret_cast<const float4 *>(ckpt) + i);
}

template <int N>
__global__ void requant_kernel(const void *ckpt, int f16, uint8_t *q, float *scale, long long n4) {
    constexpr int G4 = N / 4;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool in = i < n4;
    const float4 h = in ? ckpt_load4(ckpt, i, f16) : make_float4(0, 0, 0, 0);
    float m = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
    m = group_max<G4>(m);
    float sc, inv;
    e4m3_row_scale(m, sc, inv);
    if (!in) return;
    reinterpret_cast<uint32_t *>(q)[i] =
        e4m3_pack4(__fmul_rn(h.x, inv), __fmul_rn(h.y, inv), __fmul_rn(h.z, inv), __fmul_rn(h.w, inv));
    if ((threadIdx.x & (G4 - 1)) == 0) scale[i / G4] = sc;
}

// NVFP4 copy: the same thread mapping; a 16-column block spans 4 lanes.
template <int N>
__global__ void requant_nv4_kernel(const void *ckpt, int f16, uint8_t *q, float *scale, long long n4, int P) {
    constexpr int G4 = N / 4;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool in = i < n4;
    const float4 h = in ? ckpt_load4(ckpt, i, f16) : make_float4(0, 0, 0, 0);
    const float m4 = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
    const float m = group_max<G4>(m4), mb = group_max<4>(m4);
    float s_r, k_r, inv;
    nv4_row_scale(m, s_r, k_r);
    const uint32_t sb = nv4_block_scale(mb, s_r, k_r, inv);
    if (!in) return;
    const long long row = i / G4, head = row / P;
    const int p = (int)(row - head * P), col4 = (int)(i - row * G4);
    uint8_t *hq = q + head * nv4_head_bytes(P, N);
    reinterpret_cast<uint16_t *>(hq + p * (N / 2))[col4] =
        (uint16_t)e2m1_pack4(__fmul_rn(h.x, inv), __fmul_rn(h.y, inv), __fmul_rn(h.z, inv), __fmul_rn(h.w, inv));
    if ((col4 & 3) == 0) hq[P * N / 2 + p * (N / 16) + col4 / 4] = (uint8_t)sb;
    if (col4 == 0) scale[row] = s_r;
}

}  // namespace

// Rollback of ring_len by T - accepted[b] on the device (Mamba-2 and GDN caches
// share the ring metadata).
rssm_status launch_ring_rollback(int batch, int L, int T, const int32_t *accepted, const int32_t *slots, int cap,
                                 int32_t *ring_head, int32_t *ring_len, uint32_t *err, cudaStream_t st) {
    const int thr = 128;
    rollback_kernel<<<(batch + thr - 1) / thr, thr, 0, st>>>(batch, L, T, accepted, slots, cap, ring_head,
                                                             ring_len, err);
    return launch_status();
}

}  // namespace rssm

using namespace rssm;

namespace rssm {

// Every host-side check of a replay decode call.  The no-alloc decode runs it
// with the arrival counters not yet supplied (it provides them itself, but only
// after the call is known to be valid).
rssm_status check_decode_call(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c, const float *dt,
                              const void *x, const void *B, const void *C, const float *y, bool need_arrive,
                              TileGeom *geom) {
    rssm_status s = check_dims(d);
    if (s != RSSM_OK) return s;
    if (!c) return RSSM_ERR_NULL;
    rssm_mamba2_cache probe = *c;
    if (!need_arrive && !probe.arrive) probe.arrive = reinterpret_cast<int32_t *>(16);
    if ((s = check_cache(d, &probe)) != RSSM_OK) return s;
    if (!dt || !x || !B || !C || !y) return RSSM_ERR_NULL;
    if (!aligned16(x) || !aligned16(B) || !aligned16(C)) return RSSM_ERR_ALIGN;
    if (!choose_geom(d->batch, d->nheads, d->headdim, d->dstate, *geom)) return RSSM_ERR_UNSUPPORTED;
    return RSSM_OK;
}

}  // namespace rssm

extern "C" rssm_status replayssm_decode(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c,
                                        const float *dt, const void *x, const void *B, const void *C,
                                        float *y, void *stream) {
    TileGeom g;
    rssm_status s = check_decode_call(d, c, dt, x, B, C, y, true, &g);
    if (s != RSSM_OK) return s;
    M2Args a = make_args(d, c, g);
    a.dt = dt; a.x = x; a.Bin = B; a.Cin = C; a.y = y;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // serving shapes: the persistent pipelined kernel; anything else: per tile
    s = launch_decode_persistent(d, a, st);
    if (s != RSSM_ERR_UNSUPPORTED) return s;
    return launch<kDecode, 1>(d, a, g, st);
}

extern "C" rssm_status replayssm_test_stalled_decode(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c,
                                                     const float *dt, const void *x, const void *B, const void *C,
                                                     float *y, void *stream) {
    TileGeom g;
    rssm_status s = check_decode_call(d, c, dt, x, B, C, y, true, &g);
    if (s != RSSM_OK) return s;
    M2Args a = make_args(d, c, g);
    a.dt = dt; a.x = x; a.Bin = B; a.Cin = C; a.y = y;
    return launch_decode_persistent_stalled(d, a, static_cast<cudaStream_t>(stream));
}

extern "C" rssm_status replayssm_flush(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c,
                                       const uint8_t *mask, void *stream) {
    rssm_status s = check_dims(d);
    if (s != RSSM_OK) return s;
    if ((s = check_cache(d, c)) != RSSM_OK) return s;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->headdim, d->dstate, g)) return RSSM_ERR_UNSUPPORTED;
    M2Args a = make_args(d, c, g);
    a.mask = mask;
    return launch<kFlush, 0>(d, a, g, static_cast<cudaStream_t>(stream));
}

extern "C" rssm_status replayssm_verify(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c, int32_t T,
                                        const float *dt, const void *x, const void *B, const void *C,
                                        float *y, void *stream) {
    rssm_status s = check_dims(d);
    if (s != RSSM_OK) return s;
    if ((s = check_cache(d, c)) != RSSM_OK) return s;
    if (T < 1 || T > d->L || T > kMaxT) return RSSM_ERR_RING;
    if (!dt || !x || !B || !C || !y) return RSSM_ERR_NULL;
    if (!aligned16(x) || !aligned16(B) || !aligned16(C)) return RSSM_ERR_ALIGN;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->headdim, d->dstate, g)) return RSSM_ERR_UNSUPPORTED;
    M2Args a = make_args(d, c, g);
    a.T = T; a.dt = dt; a.x = x; a.Bin = B; a.Cin = C; a.y = y;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // serving shapes: the persistent pipelined verify (+ its B/C epilogue)
    s = launch_verify_persistent(d, a, st);
    if (s != RSSM_ERR_UNSUPPORTED) return s;
    return T <= 4 ? launch<kVerify, 4>(d, a, g, st) : launch<kVerify, 8>(d, a, g, st);
}

extern "C" rssm_status replayssm_rollback(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c, int32_t T,
                                          const int32_t *accepted, void *stream) {
    rssm_status s = check_dims(d);
    if (s != RSSM_OK) return s;
    if (!c) return RSSM_ERR_NULL;
    if (!c->ring_head || !c->ring_len || !c->err || !accepted) return RSSM_ERR_NULL;
    if (T < 1 || T > d->L || T > kMaxT) return RSSM_ERR_RING;
    if (c->capacity < 0 || (!c->slots && c->capacity > 0 && c->capacity < d->batch)) return RSSM_ERR_SHAPE;
    return launch_ring_rollback(d->batch, d->L, T, accepted, c->slots, cache_capacity(d, c), c->ring_head,
                                c->ring_len, c->err, static_cast<cudaStream_t>(stream));
}

extern "C" rssm_status replayssm_requant(const rssm_mamba2_dims *d, const rssm_mamba2_cache *c,
                                         void *stream) {
    rssm_status s = check_dims(d);
    if (s != RSSM_OK) return s;
    if (!c || !c->ckpt || !c->ckpt_q || !c->ckpt_scale) return RSSM_ERR_NULL;
    if (!aligned16(c->ckpt) || !aligned16(c->ckpt_q)) return RSSM_ERR_ALIGN;
    if (c->capacity < 0) return RSSM_ERR_SHAPE;
    const long long n4 = (long long)cache_capacity(d, c) * d->nheads * d->headdim * d->dstate / 4;
    const int thr = 256;
    const long long blocks = (n4 + thr - 1) / thr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define RSSM_RQ(NN)                                                                                      \
    if (d->dstate == NN) {                                                                               \
        if (d->read_copy == 2)                                                                           \
            requant_nv4_kernel<NN><<<(unsigned)blocks, thr, 0, st>>>(c->ckpt, d->ckpt_f16, c->ckpt_q,       \
                                                                     c->ckpt_scale, n4, d->headdim);     \
        else                                                                                             \
            requant_kernel<NN><<<(unsigned)blocks, thr, 0, st>>>(c->ckpt, d->ckpt_f16, c->ckpt_q,           \
                                                                 c->ckpt_scale, n4);                     \
    }
    RSSM_RQ(16) RSSM_RQ(32) RSSM_RQ(64) RSSM_RQ(128)
#undef RSSM_RQ
    return launch_status();
}

extern "C" const char *replayssm_status_string(rssm_status s) {
    switch (s) {
        case RSSM_OK: return "ok";
        case RSSM_ERR_NULL: return "a required pointer is NULL";
        case RSSM_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case RSSM_ERR_SHAPE: return "a size is outside the supported range";
        case RSSM_ERR_RING: return "draft count outside [1, min(L, 8)]";
        case RSSM_ERR_CUDA: return "CUDA launch failed";
        case RSSM_ERR_UNSUPPORTED: return "unsupported shape combination";
    }
    return "unknown status";
}

extern "C" uint32_t replayssm_version(void) { return 0x00000100u; }
