// Gated DeltaNet (gated delta rule) decode: replay decode with the fused
// flush, standalone flush, and the conventional in-place decode.
//
// A (sequence, head) state S is dv rows of dk floats; one CTA owns R rows.
// Thread t holds float4s t, t+T, ... of the tile, so each lane keeps the same
// 4 columns for all its rows and a row's dot product with a dk-vector is a
// reduction over the dk/4 lanes of the row.
//
// Replay output from the checkpoint S_c and the records j = 0..k-1 (k-1 = the
// current token): one warp runs the backward chain u = q,
// d_j = k_j . u, u <- alpha_j (u - beta_j d_j k_j) (newest record first), which
// leaves u_0 and coefficients beta_j d_j; then o[r] = S_c[r] . u_0 +
// sum_j beta_j d_j v_j[r].  The flush folds the records into every row,
// oldest first: s <- alpha_j s + beta_j (v_j[r] - alpha_j (s . k_j)) k_j.
#include "common.cuh"
#include "gdn_fold_tc.cuh"
#include "gdn_verify_persist.cuh"
#include "host_common.h"

namespace rssm {
namespace {

enum { gDecode = 0, gFlush = 2 };

struct GArgs {
    int H, DK, DV, L, R, split, T;
    float *ckpt;
    uint16_t *rec_k, *rec_v;
    float *rec_alpha, *rec_beta;
    int32_t *ring_head, *ring_len, *arrive;
    uint32_t *err;
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    float *o;
    const uint8_t *mask;
    const int32_t *slots;   // [batch] cache slot of each batch row; nullptr: row b uses slot b
    int cap;                // sequences the cache arrays hold
};

struct GSmem {
    int al, be, coef, k, v, q, u, o, flag, total;
    __host__ __device__ GSmem(int L, int R, int DK) {
        const int KM = L + 1;
        int off = 0;
        auto take = [&off](int n) { const int at = off; off += (n + 3) & ~3; return at; };
        al = take(KM); be = take(KM); coef = take(KM);
        k = take(KM * DK); v = take(KM * R);
        q = take(DK); u = take(DK); o = take(R); flag = take(4);
        total = off;
    }
};

// 16-byte chunk of 8 bf16 -> 8 floats in shared memory
__device__ __forceinline__ void put8(float *dst, uint4 c) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    d4[0] = make_float4(bf16lo(c.x), bf16hi(c.x), bf16lo(c.y), bf16hi(c.y));
    d4[1] = make_float4(bf16lo(c.z), bf16hi(c.z), bf16lo(c.w), bf16hi(c.w));
}

template <int MODE, int DK, int VPT>
__global__ void __launch_bounds__(256) gdn_replay_kernel(const GArgs a) {
    constexpr int G4 = DK / 4;
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int b = blockIdx.y;
    const int h = blockIdx.x / a.split, sp = blockIdx.x - h * a.split;
    const int R = a.R, L = a.L, H = a.H, DV = a.DV;
    const int p0 = sp * R;
    const int sb = a.slots ? __ldg(a.slots + b) : b;           // the sequence's cache slot
    if (sb < 0 || sb >= a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.err, RSSM_DEVERR_SLOT);
        return;
    }

    const int head = a.ring_head[sb], len = a.ring_len[sb];
    if (head < 0 || head >= L || len < 0 || len > L) {
        if (blockIdx.x == 0 && tid == 0) flag_error(a.err, RSSM_DEVERR_RING_META);
        return;
    }
    if (MODE == gFlush && (len == 0 || (a.mask != nullptr && a.mask[b] == 0))) return;
    const int nrec = MODE == gDecode ? len + 1 : len;
    const bool fold = MODE == gDecode ? (len + 1 >= L) : true;

    const size_t tile = ((size_t)sb * H + h) * DV + p0;        // cache rows
    float4 *ck4 = reinterpret_cast<float4 *>(a.ckpt + tile * DK);
    float4 hv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) hv[v] = ld_stream(ck4 + tid + v * nthr);

    const GSmem lay(L, R, DK);
    float *s_al = sm + lay.al, *s_be = sm + lay.be, *s_coef = sm + lay.coef;
    float *s_k = sm + lay.k, *s_v = sm + lay.v, *s_q = sm + lay.q, *s_u = sm + lay.u, *s_o = sm + lay.o;

    // ---- stage records (ring slots for j < len, the current token at j = len)
    const size_t bh = (size_t)b * H + h, cbh = (size_t)sb * H + h;   // inputs / outputs, cache
    const int ck = DK / 8, cv = R / 8;
    const int nk = nrec * ck, nv = nrec * cv, nq = (MODE == gDecode) ? ck : 0;
    const int total = nk + nv + nq;
    for (int base = tid; base < total; base += 4 * nthr) {
        uint4 val[4];
        float *dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * nthr;
            dst[u] = nullptr;
            if (idx < total) {
                const uint16_t *src;
                if (idx < nk) {
                    const int j = idx / ck, c = idx - j * ck;
                    src = j < len ? a.rec_k + ((cbh * L + (head + j) % L) * DK + c * 8) : a.k + (bh * DK + c * 8);
                    dst[u] = s_k + j * DK + c * 8;
                } else if (idx < nk + nv) {
                    const int m = idx - nk;
                    const int j = m / cv, c = m - j * cv;
                    src = j < len ? a.rec_v + ((cbh * L + (head + j) % L) * DV + p0 + c * 8)
                                  : a.v + (bh * DV + p0 + c * 8);
                    dst[u] = s_v + j * R + c * 8;
                } else {
                    const int c = idx - nk - nv;
                    src = a.q + (bh * DK + c * 8);
                    dst[u] = s_q + c * 8;
                }
                val[u] = __ldcg(reinterpret_cast<const uint4 *>(src));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (dst[u] != nullptr) put8(dst[u], val[u]);
    }
    for (int j = tid; j < nrec; j += nthr) {
        if (j < len) {
            const size_t r = cbh * L + (head + j) % L;
            s_al[j] = __ldcg(a.rec_alpha + r);
            s_be[j] = __ldcg(a.rec_beta + r);
        } else {
            s_al[j] = __ldcg(a.alpha + bh);
            s_be[j] = __ldcg(a.beta + bh);
        }
    }
    __syncthreads();

    // ---- backward chain (decode): u_0 and beta_j (k_j . u_j)
    if (MODE == gDecode && tid < 32) {
        constexpr int M = (DK + 31) / 32;
        float u[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int c = tid + 32 * m;
            u[m] = c < DK ? s_q[c] : 0.0f;
        }
        for (int j = nrec - 1; j >= 0; --j) {
            float d = 0.0f;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int c = tid + 32 * m;
                if (c < DK) d = fmaf(s_k[j * DK + c], u[m], d);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            const float cf = s_be[j] * d;
            if (tid == 0) s_coef[j] = cf;
            const float al = s_al[j];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int c = tid + 32 * m;
                if (c < DK) u[m] = al * fmaf(-cf, s_k[j * DK + c], u[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int c = tid + 32 * m;
            if (c < DK) s_u[c] = u[m];
        }
    }
    __syncthreads();

    const int col4 = tid % G4, row0 = tid / G4, rstep = nthr / G4;
    // ---- checkpoint contraction with u_0 (before the fold changes hv)
    if (MODE == gDecode) {
        const float4 u0 = *reinterpret_cast<const float4 *>(s_u + col4 * 4);
        float part[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            float d = hv[v].x * u0.x;
            d = fmaf(hv[v].y, u0.y, d);
            d = fmaf(hv[v].z, u0.z, d);
            d = fmaf(hv[v].w, u0.w, d);
            part[v] = d;
        }
        group_reduce<G4, VPT>(part);
        if (reduced_writer<G4, VPT>()) {
            constexpr int NV = (VPT <= G4) ? 1 : VPT / G4;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk) s_o[row0 + reduced_index<G4, VPT>(kk) * rstep] = part[kk];
        }
    }
    // ---- fold: sequential rank-one updates of every row, oldest record first
    if (fold) {
        for (int j = 0; j < nrec; ++j) {
            const float4 kj = *reinterpret_cast<const float4 *>(s_k + j * DK + col4 * 4);
            const float al = s_al[j], be = s_be[j];
            float d[VPT];
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                float t = hv[v].x * kj.x;
                t = fmaf(hv[v].y, kj.y, t);
                t = fmaf(hv[v].z, kj.z, t);
                t = fmaf(hv[v].w, kj.w, t);
                d[v] = t;
            }
            group_allreduce<G4, VPT>(d);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const float c = be * fmaf(-al, d[v], s_v[j * R + row0 + v * rstep]);
                hv[v].x = fmaf(c, kj.x, al * hv[v].x);
                hv[v].y = fmaf(c, kj.y, al * hv[v].y);
                hv[v].z = fmaf(c, kj.z, al * hv[v].z);
                hv[v].w = fmaf(c, kj.w, al * hv[v].w);
            }
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) st_stream(ck4 + tid + v * nthr, hv[v]);
    }
    __syncthreads();

    if (MODE == gDecode) {
        for (int r = tid; r < R; r += nthr) {
            float acc = s_o[r];
            for (int j = 0; j < nrec; ++j) acc = fmaf(s_coef[j], s_v[j * R + r], acc);
            a.o[bh * DV + p0 + r] = acc;
        }
        if (!fold) {
            const int slot = (head + len) % L;
            for (int c = tid; c < cv; c += nthr)
                *reinterpret_cast<uint4 *>(a.rec_v + (cbh * L + slot) * DV + p0 + c * 8) =
                    __ldcg(reinterpret_cast<const uint4 *>(a.v + bh * DV + p0 + c * 8));
            if (sp == 0) {
                for (int c = tid; c < ck; c += nthr)
                    *reinterpret_cast<uint4 *>(a.rec_k + (cbh * L + slot) * DK + c * 8) =
                        __ldcg(reinterpret_cast<const uint4 *>(a.k + bh * DK + c * 8));
                if (tid == 0) {
                    a.rec_alpha[cbh * L + slot] = s_al[len];
                    a.rec_beta[cbh * L + slot] = s_be[len];
                }
            }
        }
    }

    // ---- the last CTA of the sequence commits the ring pointers
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(a.arrive + sb, 1);
        if (prev == (int)gridDim.x - 1) {
            __threadfence();
            if (MODE == gDecode) {
                a.ring_head[sb] = fold ? (head + len + 1) % L : head;
                a.ring_len[sb] = fold ? 0 : len + 1;
            } else {
                a.ring_head[sb] = (head + len) % L;
                a.ring_len[sb] = 0;
            }
            a.arrive[sb] = 0;
        }
    }
}

// Speculative verify of T drafts.  Records j < len come from the ring, j = len + i is
// draft i (from the inputs).  Warp i runs draft i's backward chain from q_i at record
// len + i; every row's dot products with the T vectors u_0 are reduced once the
// checkpoint tile is in registers; a pre-flush folds the len buffered records into
// the rows (the flush's arithmetic) and stores them.  The last CTA of a sequence
// commits its ring pointers; gdn_verify_append writes the drafts' records afterwards.
struct GVSmem {
    int al, be, coef, k, v, q, u, o, total;
    __host__ __device__ GVSmem(int L, int T, int R, int DK) {
        const int KM = L + T;
        int off = 0;
        auto take = [&off](int n) { const int at = off; off += (n + 3) & ~3; return at; };
        al = take(KM); be = take(KM); coef = take(T * KM);
        k = take(KM * DK); v = take(KM * R);
        q = take(T * DK); u = take(T * DK); o = take(T * R);
        total = off;
    }
};

template <int DK, int VPT>
__global__ void __launch_bounds__(256) gdn_verify_kernel(const GArgs a) {
    constexpr int G4 = DK / 4;
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y;
    const int h = blockIdx.x / a.split, sp = blockIdx.x - h * a.split;
    const int R = a.R, L = a.L, H = a.H, DV = a.DV, T = a.T;
    const int p0 = sp * R;
    const int sb = a.slots ? __ldg(a.slots + b) : b;           // the sequence's cache slot
    if (sb < 0 || sb >= a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.err, RSSM_DEVERR_SLOT);
        return;
    }

    const int head = a.ring_head[sb], len = a.ring_len[sb];
    if (head < 0 || head >= L || len < 0 || len > L) {
        if (blockIdx.x == 0 && tid == 0) flag_error(a.err, RSSM_DEVERR_RING_META);
        return;
    }
    const bool pre = len + T > L;
    const int nrec = len + T, KM = L + T;

    const size_t tile = ((size_t)sb * H + h) * DV + p0;        // cache rows
    float4 *ck4 = reinterpret_cast<float4 *>(a.ckpt + tile * DK);
    float4 hv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) hv[v] = ld_stream(ck4 + tid + v * nthr);

    const GVSmem lay(L, T, R, DK);
    float *s_al = sm + lay.al, *s_be = sm + lay.be, *s_coef = sm + lay.coef;
    float *s_k = sm + lay.k, *s_v = sm + lay.v, *s_q = sm + lay.q, *s_u = sm + lay.u, *s_o = sm + lay.o;

    // ---- stage the records (ring slots, then the drafts) and the drafts' q
    const size_t cbh = (size_t)sb * H + h;                       // cache
    const int ck = DK / 8, cv = R / 8;
    const int nk = nrec * ck, nv = nrec * cv, nq = T * ck, total = nk + nv + nq;
    for (int idx = tid; idx < total; idx += nthr) {
        const uint16_t *src;
        float *dst;
        if (idx < nk) {
            const int j = idx / ck, c = idx - j * ck;
            src = j < len ? a.rec_k + ((cbh * L + (head + j) % L) * DK + c * 8)
                          : a.k + ((((size_t)b * T + (j - len)) * H + h) * DK + c * 8);
            dst = s_k + j * DK + c * 8;
        } else if (idx < nk + nv) {
            const int m = idx - nk, j = m / cv, c = m - j * cv;
            src = j < len ? a.rec_v + ((cbh * L + (head + j) % L) * DV + p0 + c * 8)
                          : a.v + ((((size_t)b * T + (j - len)) * H + h) * DV + p0 + c * 8);
            dst = s_v + j * R + c * 8;
        } else {
            const int m = idx - nk - nv, i = m / ck, c = m - i * ck;
            src = a.q + ((((size_t)b * T + i) * H + h) * DK + c * 8);
            dst = s_q + i * DK + c * 8;
        }
        put8(dst, __ldcg(reinterpret_cast<const uint4 *>(src)));
    }
    for (int j = tid; j < nrec; j += nthr) {
        if (j < len) {
            const size_t r = cbh * L + (head + j) % L;
            s_al[j] = __ldcg(a.rec_alpha + r);
            s_be[j] = __ldcg(a.rec_beta + r);
        } else {
            const size_t r = ((size_t)b * T + (j - len)) * H + h;
            s_al[j] = __ldcg(a.alpha + r);
            s_be[j] = __ldcg(a.beta + r);
        }
    }
    __syncthreads();

    // ---- backward chains, one warp per draft: u_0 and beta_j (k_j . u_j)
    for (int i = warp; i < T; i += nthr / 32) {
        constexpr int M = (DK + 31) / 32;
        float u[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int c = lane + 32 * m;
            u[m] = c < DK ? s_q[i * DK + c] : 0.0f;
        }
        for (int j = len + i; j >= 0; --j) {
            float d = 0.0f;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int c = lane + 32 * m;
                if (c < DK) d = fmaf(s_k[j * DK + c], u[m], d);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            const float cf = s_be[j] * d;
            if (lane == 0) s_coef[i * KM + j] = cf;
            const float al = s_al[j];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int c = lane + 32 * m;
                if (c < DK) u[m] = al * fmaf(-cf, s_k[j * DK + c], u[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int c = lane + 32 * m;
            if (c < DK) s_u[i * DK + c] = u[m];
        }
    }
    __syncthreads();

    // ---- checkpoint contraction with every draft's u_0 (before a pre-flush changes hv)
    const int col4 = tid % G4, row0 = tid / G4, rstep = nthr / G4;
    for (int i = 0; i < T; ++i) {
        const float4 u0 = *reinterpret_cast<const float4 *>(s_u + i * DK + col4 * 4);
        float part[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            float d = hv[v].x * u0.x;
            d = fmaf(hv[v].y, u0.y, d);
            d = fmaf(hv[v].z, u0.z, d);
            d = fmaf(hv[v].w, u0.w, d);
            part[v] = d;
        }
        group_reduce<G4, VPT>(part);
        if (reduced_writer<G4, VPT>()) {
            constexpr int NV = (VPT <= G4) ? 1 : VPT / G4;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk) s_o[i * R + row0 + reduced_index<G4, VPT>(kk) * rstep] = part[kk];
        }
    }
    // ---- pre-flush: fold the len buffered records into every row, oldest first
    if (pre) {
        for (int j = 0; j < len; ++j) {
            const float4 kj = *reinterpret_cast<const float4 *>(s_k + j * DK + col4 * 4);
            const float al = s_al[j], be = s_be[j];
            float d[VPT];
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                float t = hv[v].x * kj.x;
                t = fmaf(hv[v].y, kj.y, t);
                t = fmaf(hv[v].z, kj.z, t);
                t = fmaf(hv[v].w, kj.w, t);
                d[v] = t;
            }
            group_allreduce<G4, VPT>(d);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const float c = be * fmaf(-al, d[v], s_v[j * R + row0 + v * rstep]);
                hv[v].x = fmaf(c, kj.x, al * hv[v].x);
                hv[v].y = fmaf(c, kj.y, al * hv[v].y);
                hv[v].z = fmaf(c, kj.z, al * hv[v].z);
                hv[v].w = fmaf(c, kj.w, al * hv[v].w);
            }
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) st_stream(ck4 + tid + v * nthr, hv[v]);
    }
    __syncthreads();

    // ---- outputs: o_i[r] = S_c[r] . u_0(i) + sum_{j <= len + i} coef_ij v_j[r]
    for (int idx = tid; idx < T * R; idx += nthr) {
        const int i = idx / R, r = idx - i * R;
        float acc = s_o[i * R + r];
        for (int j = 0; j <= len + i; ++j) acc = fmaf(s_coef[i * KM + j], s_v[j * R + r], acc);
        a.o[(((size_t)b * T + i) * H + h) * DV + p0 + r] = acc;
    }

    // ---- the last CTA of the sequence commits its ring pointers
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(a.arrive + sb, 1) == (int)gridDim.x - 1) {
            __threadfence();
            a.ring_head[sb] = pre ? (head + len) % L : head;
            a.ring_len[sb] = (pre ? 0 : len) + T;
            a.arrive[sb] = 0;
        }
    }
}

// After gdn_verify_kernel: the T drafts' records of every (sequence, head) go to
// the last T slots of the ring, whose pointers the verify has committed.
__global__ void gdn_verify_append(const GArgs a) {
    const int bh = blockIdx.x, b = bh / a.H, h = bh - b * a.H;
    const int sb = a.slots ? __ldg(a.slots + b) : b;           // (the verify flagged a bad slot)
    if (sb < 0 || sb >= a.cap) return;
    const int hd = a.ring_head[sb], ln = a.ring_len[sb], L = a.L, T = a.T, DK = a.DK, DV = a.DV;
    if (hd < 0 || hd >= L || ln < T || ln > L) return;
    const int ck = DK / 8, cv = DV / 8;
    for (int idx = threadIdx.x; idx < T * (ck + cv + 1); idx += blockDim.x) {
        const int i = idx / (ck + cv + 1), c = idx - i * (ck + cv + 1);
        const int slot = (hd + ln - T + i) % L;
        const size_t src = ((size_t)b * T + i) * a.H + h, dst = ((size_t)sb * a.H + h) * L + slot;
        if (c < ck) {
            *reinterpret_cast<uint4 *>(a.rec_k + dst * DK + c * 8) =
                __ldcg(reinterpret_cast<const uint4 *>(a.k + src * DK + c * 8));
        } else if (c < ck + cv) {
            *reinterpret_cast<uint4 *>(a.rec_v + dst * DV + (c - ck) * 8) =
                __ldcg(reinterpret_cast<const uint4 *>(a.v + src * DV + (c - ck) * 8));
        } else {
            a.rec_alpha[dst] = __ldcg(a.alpha + src);
            a.rec_beta[dst] = __ldcg(a.beta + src);
        }
    }
}

// Conventional in-place step: per row d = s . k; s <- alpha s + beta (v_r -
// alpha d) k; o_r = s . q.
template <int DK, int VPT>
__global__ void __launch_bounds__(256) gdn_conv_kernel(const GArgs a) {
    constexpr int G4 = DK / 4;
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int b = blockIdx.y;
    const int h = blockIdx.x / a.split, sp = blockIdx.x - h * a.split;
    const int R = a.R, DV = a.DV;
    const int p0 = sp * R;
    const size_t bh = (size_t)b * a.H + h;
    float4 *ck4 = reinterpret_cast<float4 *>(a.ckpt + (bh * DV + p0) * DK);
    float4 hv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) hv[v] = ld_stream(ck4 + tid + v * nthr);
    float *s_k = sm, *s_q = sm + DK, *s_v = sm + 2 * DK, *s_o = s_v + R;
    for (int c = tid; c < (2 * DK + R) / 8; c += nthr) {
        const uint16_t *src;
        float *dst;
        if (c < DK / 8) { src = a.k + bh * DK + c * 8; dst = s_k + c * 8; }
        else if (c < 2 * DK / 8) { src = a.q + bh * DK + (c - DK / 8) * 8; dst = s_q + (c - DK / 8) * 8; }
        else { src = a.v + bh * DV + p0 + (c - 2 * DK / 8) * 8; dst = s_v + (c - 2 * DK / 8) * 8; }
        put8(dst, __ldcg(reinterpret_cast<const uint4 *>(src)));
    }
    __syncthreads();
    const float al = a.alpha[bh], be = a.beta[bh];
    const int col4 = tid % G4, row0 = tid / G4, rstep = nthr / G4;
    const float4 kk = *reinterpret_cast<const float4 *>(s_k + col4 * 4);
    const float4 qq = *reinterpret_cast<const float4 *>(s_q + col4 * 4);
    float d[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        float t = hv[v].x * kk.x;
        t = fmaf(hv[v].y, kk.y, t);
        t = fmaf(hv[v].z, kk.z, t);
        t = fmaf(hv[v].w, kk.w, t);
        d[v] = t;
    }
    group_allreduce<G4, VPT>(d);
    float part[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const float c = be * fmaf(-al, d[v], s_v[row0 + v * rstep]);
        hv[v].x = fmaf(c, kk.x, al * hv[v].x);
        hv[v].y = fmaf(c, kk.y, al * hv[v].y);
        hv[v].z = fmaf(c, kk.z, al * hv[v].z);
        hv[v].w = fmaf(c, kk.w, al * hv[v].w);
        st_stream(ck4 + tid + v * nthr, hv[v]);
        float t = hv[v].x * qq.x;
        t = fmaf(hv[v].y, qq.y, t);
        t = fmaf(hv[v].z, qq.z, t);
        t = fmaf(hv[v].w, qq.w, t);
        part[v] = t;
    }
    group_reduce<G4, VPT>(part);
    if (reduced_writer<G4, VPT>()) {
        constexpr int NV = (VPT <= G4) ? 1 : VPT / G4;
#pragma unroll
        for (int i = 0; i < NV; ++i) s_o[row0 + reduced_index<G4, VPT>(i) * rstep] = part[i];
    }
    __syncthreads();
    for (int r = tid; r < R; r += nthr) a.o[bh * DV + p0 + r] = s_o[r];
}

rssm_status check(const rssm_gdn_dims *d) {
    if (!d) return RSSM_ERR_NULL;
    if (d->batch < 1 || d->batch > 65535 || d->nheads < 1) return RSSM_ERR_SHAPE;
    if (!(d->dk == 16 || d->dk == 32 || d->dk == 64 || d->dk == 128)) return RSSM_ERR_SHAPE;
    if (d->dv < 8 || d->dv > 256 || d->dv % 8) return RSSM_ERR_SHAPE;
    if (d->L < 1 || d->L > kMaxL) return RSSM_ERR_SHAPE;
    return RSSM_OK;
}

rssm_status check_cache(const rssm_gdn_dims *d, const rssm_gdn_cache *c) {
    if (!c) return RSSM_ERR_NULL;
    if (!c->ckpt || !c->rec_k || !c->rec_v || !c->rec_alpha || !c->rec_beta || !c->ring_head ||
        !c->ring_len || !c->arrive || !c->err)
        return RSSM_ERR_NULL;
    if (!aligned16(c->ckpt) || !aligned16(c->rec_k) || !aligned16(c->rec_v)) return RSSM_ERR_ALIGN;
    if (c->capacity < 0 || (!c->slots && c->capacity > 0 && c->capacity < d->batch)) return RSSM_ERR_SHAPE;
    return RSSM_OK;
}

int cache_capacity(const rssm_gdn_dims *d, const rssm_gdn_cache *c) {
    return c->capacity > 0 ? c->capacity : d->batch;
}

template <int MODE>
void *pick_replay(int DK, int vpt) {
#define RSSM_PICK(NN) \
    if (DK == NN) return vpt == 8 ? (void *)gdn_replay_kernel<MODE, NN, 8> : (void *)gdn_replay_kernel<MODE, NN, 2>;
    RSSM_PICK(16) RSSM_PICK(32) RSSM_PICK(64) RSSM_PICK(128)
#undef RSSM_PICK
    return nullptr;
}

void *pick_verify(int DK, int vpt) {
#define RSSM_PICK(NN) \
    if (DK == NN) return vpt == 8 ? (void *)gdn_verify_kernel<NN, 8> : (void *)gdn_verify_kernel<NN, 2>;
    RSSM_PICK(16) RSSM_PICK(32) RSSM_PICK(64) RSSM_PICK(128)
#undef RSSM_PICK
    return nullptr;
}

void *pick_conv(int DK, int vpt) {
#define RSSM_PICK(NN) \
    if (DK == NN) return vpt == 8 ? (void *)gdn_conv_kernel<NN, 8> : (void *)gdn_conv_kernel<NN, 2>;
    RSSM_PICK(16) RSSM_PICK(32) RSSM_PICK(64) RSSM_PICK(128)
#undef RSSM_PICK
    return nullptr;
}

GArgs make_args(const rssm_gdn_dims *d, const TileGeom &g) {
    GArgs a{};
    a.H = d->nheads; a.DK = d->dk; a.DV = d->dv; a.L = d->L; a.R = g.R; a.split = g.split;
    return a;
}

void set_cache(GArgs &a, const rssm_gdn_dims *d, const rssm_gdn_cache *c) {
    a.ckpt = c->ckpt; a.rec_k = c->rec_k; a.rec_v = c->rec_v; a.rec_alpha = c->rec_alpha;
    a.rec_beta = c->rec_beta; a.ring_head = c->ring_head; a.ring_len = c->ring_len;
    a.arrive = c->arrive; a.err = c->err;
    a.slots = c->slots; a.cap = cache_capacity(d, c);
}

rssm_status launch(void *k, const rssm_gdn_dims *d, GArgs &a, const TileGeom &g, size_t smem,
                   cudaStream_t st) {
    if (!k) return RSSM_ERR_UNSUPPORTED;
    rssm_status s = ensure_smem((const void *)k, smem);
    if (s != RSSM_OK) return s;
    void *params[] = {&a};
    if (cudaLaunchKernel(k, dim3(d->nheads * g.split, d->batch), dim3(g.threads), params, smem, st) !=
        cudaSuccess)
        return RSSM_ERR_CUDA;
    return launch_status();
}

// Persistent verify at the serving head shape (dk = dv = 128, T <= 4, L <= 16)
// when every SM gets at least two items; RSSM_ERR_UNSUPPORTED (nothing launched)
// otherwise.
rssm_status launch_verify_persistent(const rssm_gdn_dims *d, const rssm_gdn_cache *c, int T, const uint16_t *q,
                                     const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                                     float *o, cudaStream_t st) {
    if (d->dk != 128 || d->dv != 128 || d->L > kGdnMaxL || T > kGdnVT) return RSSM_ERR_UNSUPPORTED;
    const int sms = sm_count();
    const long long items = (long long)d->batch * d->nheads;
    if (items < 2LL * sms || items > (1LL << 30)) return RSSM_ERR_UNSUPPORTED;
    const int grid = sms;
    const int max_my = (int)((items + grid - 1) / grid);
    if (max_my > 4096) return RSSM_ERR_UNSUPPORTED;
    constexpr int RB = 4;
    int stages = 0;
    size_t smem = 0;
    for (int s = 6; s >= 2; --s) {
        const GVPSmem lay(128, 128, d->L, T, s, RB, max_my);
        if (lay.total <= 227 * 1024) { stages = s; smem = lay.total; break; }
    }
    if (!stages) return RSSM_ERR_UNSUPPORTED;
    GPArgs a{};
    a.H = d->nheads; a.L = d->L; a.items = (int)items; a.max_my = max_my; a.stages = stages; a.recbufs = RB;
    a.T = T;
    a.ckpt = c->ckpt; a.rec_k = c->rec_k; a.rec_v = c->rec_v; a.rec_alpha = c->rec_alpha; a.rec_beta = c->rec_beta;
    a.ring_head = c->ring_head; a.ring_len = c->ring_len; a.arrive = c->arrive; a.err = c->err;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.o = o;
    a.slots = c->slots; a.cap = cache_capacity(d, c);
    void *kern = (void *)gdn_verify_persistent<128, 128>;
    rssm_status s = ensure_smem((const void *)kern, smem);
    if (s != RSSM_OK) return s;
    void *params[] = {&a};
    if (cudaLaunchKernel(kern, dim3(grid), dim3(256 + 64 + kPrepThreads), params, smem, st) != cudaSuccess)
        return RSSM_ERR_CUDA;
    return launch_status();
}

// Persistent decode at the serving head shape (dk = dv = 128) when every SM
// gets at least two items; RSSM_ERR_UNSUPPORTED (nothing launched) otherwise.
rssm_status launch_persistent(const rssm_gdn_dims *d, const rssm_gdn_cache *c, const uint16_t *q,
                              const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                              float *o, cudaStream_t st) {
    if (d->dk != 128 || d->dv != 128 || d->L > kGdnMaxL) return RSSM_ERR_UNSUPPORTED;
    const int sms = sm_count();
    const long long items = (long long)d->batch * d->nheads;
    if (items < 2LL * sms || items > (1LL << 30)) return RSSM_ERR_UNSUPPORTED;
    const int grid = sms;
    const int max_my = (int)((items + grid - 1) / grid);
    if (max_my > 4096) return RSSM_ERR_UNSUPPORTED;
    constexpr int RB = 4;                                // even: each preparation warp keeps its own buffers
    // the folding items go to the tensor-core fold phase when its shared memory
    // plan fits next to the per-item lists; otherwise the decode phase folds them
    int stages = 0;
    size_t smem = 0;
    bool fold_phase = max_my <= kFtMaxMy;
    for (int pass = 0; pass < 2 && !stages; ++pass, fold_phase = false) {
        for (int s = 6; s >= 2; --s) {
            const GStepSmem lay(d->L, s, RB, max_my, fold_phase);
            if (lay.total <= 227 * 1024) { stages = s; smem = lay.total; break; }
        }
        if (stages) break;
    }
    if (!stages) return RSSM_ERR_UNSUPPORTED;
    GPArgs a{};
    a.H = d->nheads; a.L = d->L; a.items = (int)items; a.max_my = max_my; a.stages = stages; a.recbufs = RB;
    a.ckpt = c->ckpt; a.rec_k = c->rec_k; a.rec_v = c->rec_v; a.rec_alpha = c->rec_alpha; a.rec_beta = c->rec_beta;
    a.ring_head = c->ring_head; a.ring_len = c->ring_len; a.arrive = c->arrive; a.err = c->err;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.o = o;
    a.slots = c->slots; a.cap = cache_capacity(d, c);
    a.skip_folds = fold_phase ? 1 : 0;
    void *kern = (void *)gdn_decode_persistent<128, 128>;
    rssm_status s = ensure_smem((const void *)kern, smem);
    if (s != RSSM_OK) return s;
    void *params[] = {&a};
    if (cudaLaunchKernel(kern, dim3(grid), dim3(256 + 64 + kPrepThreads), params, smem, st) != cudaSuccess)
        return RSSM_ERR_CUDA;
    return launch_status();
}

}  // namespace
}  // namespace rssm

using namespace rssm;

extern "C" rssm_status replayssm_gdn_decode(const rssm_gdn_dims *d, const rssm_gdn_cache *c, const uint16_t *q,
                                            const uint16_t *k, const uint16_t *v, const float *alpha,
                                            const float *beta, float *o, void *stream) {
    rssm_status s = check(d);
    if (s != RSSM_OK) return s;
    if ((s = check_cache(d, c)) != RSSM_OK) return s;
    if (!q || !k || !v || !alpha || !beta || !o) return RSSM_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return RSSM_ERR_ALIGN;
    s = launch_persistent(d, c, q, k, v, alpha, beta, o, static_cast<cudaStream_t>(stream));
    if (s != RSSM_ERR_UNSUPPORTED) return s;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->dv, d->dk, g)) return RSSM_ERR_UNSUPPORTED;
    GArgs a = make_args(d, g);
    set_cache(a, d, c);
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.o = o;
    const size_t smem = (size_t)GSmem(d->L, g.R, d->dk).total * sizeof(float);
    return launch(pick_replay<gDecode>(d->dk, g.vpt), d, a, g, smem, static_cast<cudaStream_t>(stream));
}

extern "C" rssm_status replayssm_gdn_flush(const rssm_gdn_dims *d, const rssm_gdn_cache *c, const uint8_t *mask,
                                           void *stream) {
    rssm_status s = check(d);
    if (s != RSSM_OK) return s;
    if ((s = check_cache(d, c)) != RSSM_OK) return s;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->dv, d->dk, g)) return RSSM_ERR_UNSUPPORTED;
    GArgs a = make_args(d, g);
    set_cache(a, d, c);
    a.mask = mask;
    const size_t smem = (size_t)GSmem(d->L, g.R, d->dk).total * sizeof(float);
    return launch(pick_replay<gFlush>(d->dk, g.vpt), d, a, g, smem, static_cast<cudaStream_t>(stream));
}

extern "C" rssm_status replayssm_gdn_verify(const rssm_gdn_dims *d, const rssm_gdn_cache *c, int32_t T,
                                            const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                            const float *alpha, const float *beta, float *o, void *stream) {
    rssm_status s = check(d);
    if (s != RSSM_OK) return s;
    if ((s = check_cache(d, c)) != RSSM_OK) return s;
    if (T < 1 || T > kMaxT || T > d->L) return RSSM_ERR_RING;
    if (!q || !k || !v || !alpha || !beta || !o) return RSSM_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return RSSM_ERR_ALIGN;
    // serving shapes: the persistent pipelined verify (it appends the drafts itself)
    s = launch_verify_persistent(d, c, T, q, k, v, alpha, beta, o, static_cast<cudaStream_t>(stream));
    if (s != RSSM_ERR_UNSUPPORTED) return s;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->dv, d->dk, g)) return RSSM_ERR_UNSUPPORTED;
    GArgs a = make_args(d, g);
    set_cache(a, d, c);
    a.T = T; a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.o = o;
    const size_t smem = (size_t)GVSmem(d->L, T, g.R, d->dk).total * sizeof(float);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = launch(pick_verify(d->dk, g.vpt), d, a, g, smem, st)) != RSSM_OK) return s;
    gdn_verify_append<<<d->batch * d->nheads, 128, 0, st>>>(a);
    return launch_status();
}

extern "C" rssm_status replayssm_gdn_rollback(const rssm_gdn_dims *d, const rssm_gdn_cache *c, int32_t T,
                                              const int32_t *accepted, void *stream) {
    rssm_status s = check(d);
    if (s != RSSM_OK) return s;
    if (!c || !c->ring_head || !c->ring_len || !c->err || !accepted) return RSSM_ERR_NULL;
    if (T < 1 || T > kMaxT || T > d->L) return RSSM_ERR_RING;
    if (c->capacity < 0 || (!c->slots && c->capacity > 0 && c->capacity < d->batch)) return RSSM_ERR_SHAPE;
    return rssm::launch_ring_rollback(d->batch, d->L, T, accepted, c->slots, cache_capacity(d, c), c->ring_head,
                                      c->ring_len,
                                      c->err, static_cast<cudaStream_t>(stream));
}

extern "C" rssm_status replayssm_gdn_conventional_decode(const rssm_gdn_dims *d, float *state, const uint16_t *q,
                                                         const uint16_t *k, const uint16_t *v, const float *alpha,
                                                         const float *beta, float *o, void *stream) {
    rssm_status s = check(d);
    if (s != RSSM_OK) return s;
    if (!state || !q || !k || !v || !alpha || !beta || !o) return RSSM_ERR_NULL;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return RSSM_ERR_ALIGN;
    TileGeom g;
    if (!choose_geom(d->batch, d->nheads, d->dv, d->dk, g)) return RSSM_ERR_UNSUPPORTED;
    GArgs a = make_args(d, g);
    a.ckpt = state; a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.o = o;
    const size_t smem = ((size_t)2 * d->dk + 2 * g.R + 4) * sizeof(float);
    return launch(pick_conv(d->dk, g.vpt), d, a, g, smem, static_cast<cudaStream_t>(stream));
}
