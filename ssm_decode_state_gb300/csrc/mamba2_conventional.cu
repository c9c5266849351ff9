// Conventional Mamba-2 decode paths kept for comparison: the in-place decode
// step that loads, updates and stores the whole state every token, and the
// speculative verify that stores a state snapshot after every draft.
//
// Same tile mapping as the replay kernels: one CTA per R rows of a (sequence,
// head) state, VPT float4 per thread, the N/4 lanes of a row reduce its dot
// product with C.
#include "common.cuh"
#include "host_common.h"

namespace rssm {
namespace {

struct ConvArgs {
    int H, P, N, G, R, split, T, hpg, io_bf16;
    float *state;            // [b][H][P][N] or pool [b][T+1][H][P][N]
    const int32_t *slot;     // verify: pool entry of the current state
    const float *A, *D, *dt;
    const void *x, *Bin, *Cin;
    float *y;
    uint32_t *err;
};

// Stage Q tokens' x rows (R), B and C rows (N) into shared memory as float32.
// Token i's inputs: x at element offset xrow(i), B/C at brow(i).
template <typename XRow, typename BRow>
__device__ void stage_tokens(int Q, int R, int N, int p0, bool bf, const void *x, const void *Bin,
                             const void *Cin, XRow xrow, BRow brow, float *s_x, float *s_B, float *s_C) {
    const int E = bf ? 8 : 4, esz = bf ? 2 : 4;
    const int cx = R / E, cB = N / E;
    const int total = Q * (cx + 2 * cB);
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const char *src;
        float *dst;
        if (idx < Q * cx) {
            const int i = idx / cx, c = idx - i * cx;
            src = static_cast<const char *>(x) + ((size_t)xrow(i) + p0 + c * E) * esz;
            dst = s_x + i * R + c * E;
        } else {
            const int k = idx - Q * cx;
            const bool isC = k >= Q * cB;
            const int kk = isC ? k - Q * cB : k;
            const int i = kk / cB, c = kk - i * cB;
            src = static_cast<const char *>(isC ? Cin : Bin) + ((size_t)brow(i) + c * E) * esz;
            dst = (isC ? s_C : s_B) + i * N + c * E;
        }
        float f[8];
        unpack_chunk(__ldcg(reinterpret_cast<const uint4 *>(src)), bf, f);
        float4 *d4 = reinterpret_cast<float4 *>(dst);
        d4[0] = make_float4(f[0], f[1], f[2], f[3]);
        if (bf) d4[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
}

// Q = 1: in-place decode.  Q = T (<= TQ): snapshot verify.
template <int N, int VPT, int TQ>
__global__ void __launch_bounds__(256) m2_conv_kernel(const ConvArgs a) {
    constexpr int G4 = N / 4;
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int b = blockIdx.y;
    const int h = blockIdx.x / a.split, sp = blockIdx.x - h * a.split;
    const int g = h / a.hpg;
    const int R = a.R, N_ = a.N, P = a.P, H = a.H;
    const int p0 = sp * R;
    const bool verify = a.T > 0;
    const int Q = verify ? a.T : 1;
    const int nslot = a.T + 1;

    int cur = 0;
    if (verify) {
        cur = a.slot[b];
        if (cur < 0 || cur >= nslot) {
            if (blockIdx.x == 0 && tid == 0) flag_error(a.err, RSSM_DEVERR_SLOT);
            return;
        }
    }
    // state tile of pool entry e
    auto tile_ptr = [&](int e) -> float4 * {
        const size_t ent = verify ? ((size_t)b * nslot + e) : (size_t)b;
        return reinterpret_cast<float4 *>(a.state + ((ent * H + h) * P + p0) * (size_t)N_);
    };
    float4 hv[VPT];
    {
        const float4 *src = tile_ptr(cur);
#pragma unroll
        for (int v = 0; v < VPT; ++v) hv[v] = ld_stream(src + tid + v * nthr);
    }

    float *s_x = sm;                      // [TQ][R]
    float *s_B = s_x + TQ * R;            // [TQ][N]
    float *s_C = s_B + TQ * N;            // [TQ][N]
    float *s_y = s_C + TQ * N;            // [TQ][R]
    float *s_dt = s_y + TQ * R;           // [TQ]
    const bool bf = a.io_bf16 != 0;
    auto xrow = [&](int i) -> size_t {
        return (verify ? (((size_t)b * a.T + i) * H + h) : ((size_t)b * H + h)) * P;
    };
    auto brow = [&](int i) -> size_t {
        return (verify ? (((size_t)b * a.T + i) * a.G + g) : ((size_t)b * a.G + g)) * N_;
    };
    stage_tokens(Q, R, N_, p0, bf, a.x, a.Bin, a.Cin, xrow, brow, s_x, s_B, s_C);
    for (int i = tid; i < Q; i += nthr)
        s_dt[i] = verify ? a.dt[((size_t)b * a.T + i) * H + h] : a.dt[(size_t)b * H + h];
    __syncthreads();

    const float Ah = a.A[h], Dh = a.D[h];
    const int col4 = tid % G4, row0 = tid / G4, rstep = nthr / G4;
    float part[TQ * VPT];
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
        if (i < Q) {
            const float d = s_dt[i];
            const float dec = expf(d * Ah);
            const float4 Bi = *reinterpret_cast<const float4 *>(s_B + i * N + col4 * 4);
            const float4 Ci = *reinterpret_cast<const float4 *>(s_C + i * N + col4 * 4);
            float4 *dst = verify ? tile_ptr((cur + 1 + i) % nslot) : tile_ptr(0);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                // one rounding of the state per step: the small input term is
                // formed first, the decayed state is added in one fma
                const float dx = d * s_x[i * R + row0 + v * rstep];
                hv[v].x = fmaf(dec, hv[v].x, dx * Bi.x);
                hv[v].y = fmaf(dec, hv[v].y, dx * Bi.y);
                hv[v].z = fmaf(dec, hv[v].z, dx * Bi.z);
                hv[v].w = fmaf(dec, hv[v].w, dx * Bi.w);
                st_stream(dst + tid + v * nthr, hv[v]);
                float s = hv[v].x * Ci.x;
                s = fmaf(hv[v].y, Ci.y, s);
                s = fmaf(hv[v].z, Ci.z, s);
                s = fmaf(hv[v].w, Ci.w, s);
                part[i * VPT + v] = s;
            }
        } else {
#pragma unroll
            for (int v = 0; v < VPT; ++v) part[i * VPT + v] = 0.0f;
        }
    }
    group_reduce<G4, TQ * VPT>(part);
    if (reduced_writer<G4, TQ * VPT>()) {
        constexpr int NV = (TQ * VPT <= G4) ? 1 : (TQ * VPT) / G4;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = reduced_index<G4, TQ * VPT>(k);
            const int i = vi / VPT, v = vi - i * VPT;
            if (i < Q) s_y[i * R + row0 + v * rstep] = part[k];
        }
    }
    __syncthreads();
    for (int idx = tid; idx < Q * R; idx += nthr) {
        const int i = idx / R, r = idx - i * R;
        const size_t yrow = verify ? (((size_t)b * a.T + i) * H + h) : ((size_t)b * H + h);
        a.y[yrow * P + p0 + r] = fmaf(Dh, s_x[idx], s_y[idx]);
    }
}

__global__ void select_kernel(int batch, int T, int32_t *slot, const int32_t *accepted, uint32_t *err) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int s = slot[b], acc = accepted[b];
    if (s < 0 || s > T) {
        flag_error(err, RSSM_DEVERR_SLOT);
        return;
    }
    if (acc < 0 || acc > T) {
        flag_error(err, RSSM_DEVERR_ROLLBACK);
        return;
    }
    slot[b] = (s + acc) % (T + 1);
}

rssm_status check(const rssm_mamba2_dims *d) {
    if (!d) return RSSM_ERR_NULL;
    if (d->batch < 1 || d->batch > 65535 || d->nheads < 1 || d->ngroups < 1 || d->nheads % d->ngroups)
        return RSSM_ERR_SHAPE;
    if (!(d->dstate == 16 || d->dstate == 32 || d->dstate == 64 || d->dstate == 128)) return RSSM_ERR_SHAPE;
    if (d->headdim < 8 || d->headdim > 256 || d->headdim % 8) return RSSM_ERR_SHAPE;
    if (d->io_bf16 != 0 && d->io_bf16 != 1) return RSSM_ERR_SHAPE;
    return RSSM_OK;
}

template <int TQ>
void *pick(int N, int vpt) {
#define RSSM_PICK(NN)                                                                   \
    if (N == NN) return vpt == 8 ? (void *)m2_conv_kernel<NN, 8, TQ> : (void *)m2_conv_kernel<NN, 2, TQ>;
    RSSM_PICK(16) RSSM_PICK(32) RSSM_PICK(64) RSSM_PICK(128)
#undef RSSM_PICK
    return nullptr;
}

template <int TQ>
rssm_status launch(const rssm_mamba2_dims *d, ConvArgs &a, const TileGeom &g, cudaStream_t st) {
    void *k = pick<TQ>(d->dstate, g.vpt);
    if (!k) return RSSM_ERR_UNSUPPORTED;
    const size_t smem = ((size_t)TQ * (2 * g.R + 2 * d->dstate) + TQ + 4) * sizeof(float);
    void *params[] = {&a};
    if (cudaLaunchKernel(k, dim3(d->nheads * g.split, d->batch), dim3(g.threads), params, smem, st) !=
        cudaSuccess)
        return RSSM_ERR_CUDA;
    return launch_status();
}

}  // namespace
}  // namespace rssm

using namespace rssm;

extern "C" rssm_status replayssm_conventional_decode(const rssm_mamba2_dims *d, float *state, const float *A,
                                                     const float *D, const float *dt, const void *x,
                                                     const void *B, const void *C, float *y, void *stream) {
    rssm_status s = check(d);
    if (s != RSSM_OK) return s;
    if (!state || !A || !D || !dt || !x || !B || !C || !y) return RSSM_ERR_NULL;
    if (!aligned16(state) || !aligned16(x) || !aligned16(B) || !aligned16(C)) return RSSM_ERR_ALIGN;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->headdim, d->dstate, g)) return RSSM_ERR_UNSUPPORTED;
    ConvArgs a{};
    a.H = d->nheads; a.P = d->headdim; a.N = d->dstate; a.G = d->ngroups; a.R = g.R; a.split = g.split;
    a.T = 0; a.hpg = d->nheads / d->ngroups; a.io_bf16 = d->io_bf16;
    a.state = state; a.A = A; a.D = D; a.dt = dt; a.x = x; a.Bin = B; a.Cin = C; a.y = y;
    return launch<1>(d, a, g, static_cast<cudaStream_t>(stream));
}

extern "C" rssm_status replayssm_conventional_verify(const rssm_mamba2_dims *d, float *pool, const int32_t *slot,
                                                     int32_t T, const float *A, const float *D, const float *dt,
                                                     const void *x, const void *B, const void *C, float *y,
                                                     uint32_t *err, void *stream) {
    rssm_status s = check(d);
    if (s != RSSM_OK) return s;
    if (!pool || !slot || !A || !D || !dt || !x || !B || !C || !y || !err) return RSSM_ERR_NULL;
    if (!aligned16(pool) || !aligned16(x) || !aligned16(B) || !aligned16(C)) return RSSM_ERR_ALIGN;
    if (T < 1 || T > kMaxT) return RSSM_ERR_RING;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->headdim, d->dstate, g)) return RSSM_ERR_UNSUPPORTED;
    ConvArgs a{};
    a.H = d->nheads; a.P = d->headdim; a.N = d->dstate; a.G = d->ngroups; a.R = g.R; a.split = g.split;
    a.T = T; a.hpg = d->nheads / d->ngroups; a.io_bf16 = d->io_bf16;
    a.state = pool; a.slot = slot; a.A = A; a.D = D; a.dt = dt; a.x = x; a.Bin = B; a.Cin = C; a.y = y;
    a.err = err;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return T <= 4 ? launch<4>(d, a, g, st) : launch<8>(d, a, g, st);
}

extern "C" rssm_status replayssm_conventional_select(int32_t batch, int32_t *slot, int32_t T,
                                                     const int32_t *accepted, uint32_t *err, void *stream) {
    if (!slot || !accepted || !err) return RSSM_ERR_NULL;
    if (batch < 1) return RSSM_ERR_SHAPE;
    if (T < 1 || T > kMaxT) return RSSM_ERR_RING;
    const int thr = 128;
    select_kernel<<<(batch + thr - 1) / thr, thr, 0, static_cast<cudaStream_t>(stream)>>>(batch, T, slot,
                                                                                         accepted, err);
    return launch_status();
}
