// Mamba-2 replay kernels: decode (with the flush fused into the L-th step),
// speculative verify (with a pre-flush when the drafts would overflow the
// ring) and the standalone flush.  One template, three modes.  This is the
// per-tile kernel used for every shape; the serving shape's decode also has a
// persistent pipelined kernel (mamba2_persist.cuh).
//
// Work split.  One CTA owns the tile of R = headdim/split rows of one
// (sequence, head) checkpoint.  The tile is a flat array of float4; thread t
// holds float4s t, t+T, ..., t+(VPT-1)T.  Since T is a multiple of 32 and a
// row is N/4 float4s (N/4 divides 32), every lane keeps the same 4 columns
// for all of its rows: its 4 entries of C_t stay in registers and a row's dot
// product is a reduction over an aligned group of N/4 lanes.
//
// Per CTA:
//   0. read the ring pointers; issue the checkpoint loads (FP32 tile, or the
//      FP8 codes + row scales on a non-flush step with a read copy);
//   1. while they are in flight, stage the records into shared memory: the
//      buffered ones from the ring, the current token (or drafts) from the
//      inputs -- 16-byte loads, converted to float32;
//   2. decay weights w_j = exp(A * sum(dt after j)) dt_j and dot products
//      B_j . C_t for every (query, record) pair;
//   3. record term  sum_j w_j (B_j . C_t) x_j[p] + D x_t[p]  per row;
//   4. consume the checkpoint: fold it (flush steps) and store it back, then
//      the row dot products with C_t, reduced across the row's lanes;
//   5. y = exp(A S) (h_c . C_t) + record term; write this CTA's rows of x
//      into the ring;
//   6. arrive on the sequence's counter; the last CTA of the sequence writes
//      the records every head shares (dt, B, C) and commits the ring
//      pointers, so no CTA can overwrite a slot another one still reads.
#pragma once

#include "common.cuh"

namespace rssm {

enum { kDecode = 0, kVerify = 1, kFlush = 2 };

struct M2Args {
    int B, H, P, N, G, L, R, split, T, hpg;
    int read_copy, io_bf16;
    int ckpt_f16;                     // checkpoint in FP16 (stochastic rounding at flushes)
    uint32_t seed_lo, seed_hi;        // the call's rounding seed
    float *ckpt;                      // float32, or FP16 values when ckpt_f16
    uint8_t *ckpt_q;
    float *ckpt_scale;
    float *rec_dt;
    void *rec_x, *rec_B, *rec_C;
    int32_t *ring_head, *ring_len, *arrive;
    const int32_t *slots;   // [B] cache slot of each batch row; nullptr: row b uses slot b
    int cap;                // sequences the cache arrays hold
    const float *A, *D;
    uint32_t *err;
    const float *dt;
    const void *x, *Bin, *Cin;
    float *y;
    const uint8_t *mask;
};

// Shared-memory layout (in floats) for one CTA; the host sizes the dynamic
// allocation with the same function.
struct M2Smem {
    int dt, x, wx, Bm, C, w, cb, decay, wf, yck, rt, flag, total;
    __host__ __device__ M2Smem(int mode, int L, int T, int R, int N) {
        const int KM = L + (mode == kVerify ? T : 1);
        const int NQ = mode == kVerify ? T : (mode == kDecode ? 1 : 0);
        // every array starts on a 16-byte boundary (float4 access)
        int o = 0;
        auto take = [&o](int n) { const int at = o; o += (n + 3) & ~3; return at; };
        dt = take(KM);
        wf = take(KM + 1);               // fold weights, then the fold decay
        x = take(KM * R);
        wx = take(KM * R);
        Bm = take(KM * N);
        C = take(NQ * N);
        w = take(NQ * KM);
        cb = take(NQ * KM);
        decay = take(NQ);
        yck = take(NQ * R);
        rt = take(NQ * R);
        flag = take(4);
        total = o;
    }
};

template <int MODE, int N, int VPT, int TQ>
__global__ void __launch_bounds__(256)
m2_replay_kernel(const M2Args a) {
    constexpr int G4 = N / 4;               // lanes per row
    constexpr int NQV = (TQ > 0 ? TQ : 1);  // query slots in registers
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);

    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int b = blockIdx.y;                // batch row: inputs and outputs
    const int sb = a.slots ? a.slots[b] : b;  // cache slot of the row's sequence
    if (sb < 0 || sb >= a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.err, RSSM_DEVERR_SLOT);
        return;
    }
    const int h = blockIdx.x / a.split;
    const int sp = blockIdx.x - h * a.split;
    const int g = h / a.hpg;
    const int R = a.R, L = a.L, H = a.H, P = a.P;
    const int p0 = sp * R;
    const bool bf = a.io_bf16 != 0;
    const int E = bf ? 8 : 4;               // elements per 16-byte chunk

    // ---- 0. ring pointers and what this step does
    const int head = a.ring_head[sb];
    const int len = a.ring_len[sb];
    const bool bad = head < 0 || head >= L || len < 0 || len > L;
    if (bad) {
        if (blockIdx.x == 0 && tid == 0) flag_error(a.err, RSSM_DEVERR_RING_META);
        return;
    }
    if (MODE == kFlush && (len == 0 || (a.mask != nullptr && a.mask[b] == 0))) return;

    int nrec, nfold, nq;
    bool fold;
    if (MODE == kDecode) {
        nrec = len + 1; fold = (len + 1 >= L); nfold = fold ? nrec : 0; nq = 1;
    } else if (MODE == kVerify) {
        nrec = len + a.T; fold = (len + a.T > L); nfold = fold ? len : 0; nq = a.T;
    } else {
        nrec = len; fold = true; nfold = len; nq = 0;
    }
    const bool use_q = (MODE == kDecode) && !fold && a.read_copy;

    const M2Smem L_(MODE, L, (MODE == kVerify ? a.T : 0), R, N);
    float *s_dt = sm + L_.dt, *s_wf = sm + L_.wf, *s_x = sm + L_.x, *s_wx = sm + L_.wx;
    float *s_B = sm + L_.Bm, *s_C = sm + L_.C, *s_w = sm + L_.w, *s_cb = sm + L_.cb;
    float *s_decay = sm + L_.decay, *s_yck = sm + L_.yck, *s_rt = sm + L_.rt;
    int *s_flag = reinterpret_cast<int *>(sm + L_.flag);
    const int KM = L + (MODE == kVerify ? a.T : 1);

    // ---- checkpoint loads (in flight during staging)
    const size_t tile = ((size_t)sb * H + h) * P + p0;         // first row of the tile
    const float4 *ck4 = reinterpret_cast<const float4 *>(a.ckpt + tile * N);
    float4 hv[VPT];
    uint32_t qv[VPT];
    float qs[VPT];
    const int col4 = tid % G4;
    if (!use_q && a.ckpt_f16) {
        const uint2 *ck2 = reinterpret_cast<const uint2 *>(a.ckpt) + tile * N / 4;
#pragma unroll
        for (int v = 0; v < VPT; ++v) hv[v] = f16x4_to_float4(__ldcs(ck2 + tid + v * nthr));
    } else if (!use_q) {
#pragma unroll
        for (int v = 0; v < VPT; ++v) hv[v] = ld_stream(ck4 + tid + v * nthr);
    } else if (a.read_copy == 1) {
        const uint32_t *q4 = reinterpret_cast<const uint32_t *>(a.ckpt_q + tile * N);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            qv[v] = ld_stream_u32(q4 + tid + v * nthr);
            qs[v] = __ldcs(a.ckpt_scale + tile + (tid + v * nthr) / G4);
        }
    } else {
        // NVFP4: this thread's 4 codes of each row (16 bits) and the effective
        // scale of their block, e4m3(block scale) * row scale
        const uint8_t *hq = a.ckpt_q + ((size_t)sb * H + h) * nv4_head_bytes(P, N);
        const uint16_t *q16 = reinterpret_cast<const uint16_t *>(hq + (size_t)p0 * (N / 2));
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = tid + v * nthr, row = p0 + idx / G4;
            qv[v] = __ldcs(q16 + idx);
            qs[v] = __fmul_rn(e4m3_value(__ldcs(hq + P * N / 2 + row * (N / 16) + col4 / 4)),
                              __ldcs(a.ckpt_scale + tile + idx / G4));
        }
    }

    // ---- 1. stage records: list position j < len is ring slot (head+j) mod L,
    //         j >= len is the current token (decode) or draft j-len (verify)
    const char *rx = static_cast<const char *>(a.rec_x);
    const char *rB = static_cast<const char *>(a.rec_B);
    const char *ix = static_cast<const char *>(a.x);
    const char *iB = static_cast<const char *>(a.Bin);
    const char *iC = static_cast<const char *>(a.Cin);
    const int esz = bf ? 2 : 4;
    const int cx = R / E, cB = N / E;
    const int nx = nrec * cx, nB = nrec * cB, nC = nq * cB;
    const int total = nx + nB + nC;
    for (int base = tid; base < total; base += 4 * nthr) {
        uint4 v[4];
        float *dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * nthr;
            dst[u] = nullptr;
            if (idx < total) {
                const char *src;
                if (idx < nx) {
                    const int j = idx / cx, c = idx - j * cx;
                    if (j < len) {
                        const int slot = (head + j) % L;
                        src = rx + ((((size_t)sb * H + h) * L + slot) * P + p0 + c * E) * esz;
                    } else {
                        const int i = j - len;   // 0 for decode
                        const size_t row = MODE == kVerify ? (((size_t)b * a.T + i) * H + h)
                                                           : ((size_t)b * H + h);
                        src = ix + (row * P + p0 + c * E) * esz;
                    }
                    dst[u] = s_x + j * R + c * E;
                } else if (idx < nx + nB) {
                    const int k = idx - nx;
                    const int j = k / cB, c = k - j * cB;
                    if (j < len) {
                        const int slot = (head + j) % L;
                        src = rB + ((((size_t)sb * a.G + g) * L + slot) * N + c * E) * esz;
                    } else {
                        const int i = j - len;
                        const size_t row = MODE == kVerify ? (((size_t)b * a.T + i) * a.G + g)
                                                           : ((size_t)b * a.G + g);
                        src = iB + (row * N + c * E) * esz;
                    }
                    dst[u] = s_B + j * N + c * E;
                } else {
                    const int k = idx - nx - nB;
                    const int i = k / cB, c = k - i * cB;
                    const size_t row = MODE == kVerify ? (((size_t)b * a.T + i) * a.G + g)
                                                       : ((size_t)b * a.G + g);
                    src = iC + (row * N + c * E) * esz;
                    dst[u] = s_C + i * N + c * E;
                }
                v[u] = __ldcg(reinterpret_cast<const uint4 *>(src));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (dst[u] != nullptr) {
                float f[8];
                unpack_chunk(v[u], bf, f);
                float4 *d4 = reinterpret_cast<float4 *>(dst[u]);
                d4[0] = make_float4(f[0], f[1], f[2], f[3]);
                if (bf) d4[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }
    for (int j = tid; j < nrec; j += nthr) {
        float d;
        if (j < len) {
            d = __ldcg(a.rec_dt + ((size_t)sb * H + h) * L + (head + j) % L);
        } else {
            const int i = j - len;
            d = MODE == kVerify ? __ldcg(a.dt + ((size_t)b * a.T + i) * H + h)
                                : __ldcg(a.dt + (size_t)b * H + h);
        }
        s_dt[j] = d;
    }
    __syncthreads();

    // ---- 2. decay weights and B_j . C_i
    const float Ah = a.A[h];
    // query i reads records 0..qend(i): the checkpoint plus everything buffered
    // before it and itself
    auto qend = [&](int i) { return MODE == kVerify ? len + i : len; };
    for (int idx = tid; idx < nq * KM; idx += nthr) {
        const int i = idx / KM, j = idx - i * KM;
        const int e = qend(i);
        if (j <= e) s_w[i * KM + j] = expf(Ah * suffix_sum(s_dt, j, e)) * s_dt[j];
    }
    for (int i = tid; i < nq; i += nthr) s_decay[i] = expf(Ah * suffix_sum(s_dt, -1, qend(i)));
    if (fold) {
        for (int j = tid; j <= nfold; j += nthr) {
            s_wf[j] = (j < nfold) ? expf(Ah * suffix_sum(s_dt, j, nfold - 1)) * s_dt[j]
                                  : expf(Ah * suffix_sum(s_dt, -1, nfold - 1));
        }
    }
    {
        const int warp = tid >> 5, lane = tid & 31, nwarp = nthr >> 5;
        for (int pr = warp; pr < nq * KM; pr += nwarp) {
            const int i = pr / KM, j = pr - i * KM;
            if (j > qend(i)) continue;
            float acc = 0.0f;
            for (int n = lane; n < N; n += 32) acc = fmaf(s_B[j * N + n], s_C[i * N + n], acc);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) s_cb[i * KM + j] = acc;
        }
    }
    __syncthreads();

    // ---- 3. record term per row, fold coefficients
    const float Dh = a.D[h];
    for (int idx = tid; idx < nq * R; idx += nthr) {
        const int i = idx / R, r = idx - i * R;
        const int e = qend(i);
        float acc = 0.0f;
        for (int j = 0; j <= e; ++j)
            acc = fmaf(s_w[i * KM + j] * s_cb[i * KM + j], s_x[j * R + r], acc);
        s_rt[i * R + r] = fmaf(Dh, s_x[e * R + r], acc);
    }
    if (fold) {
        for (int idx = tid; idx < nfold * R; idx += nthr) {
            const int j = idx / R;
            s_wx[idx] = s_wf[j] * s_x[idx];
        }
    }
    __syncthreads();

    // ---- 4. consume the checkpoint tile
    const int row0 = tid / G4;              // row of v = 0 within the tile
    const int rstep = nthr / G4;            // rows between consecutive v
    if (fold) {
        const float fdec = s_wf[nfold];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int row = row0 + v * rstep;
            // rank-nfold update first, then the decayed checkpoint in one fma:
            // the state itself is rounded once per flush
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < nfold; ++j) {
                const float c = s_wx[j * R + row];
                const float4 bj = *reinterpret_cast<const float4 *>(s_B + j * N + col4 * 4);
                acc.x = fmaf(c, bj.x, acc.x);
                acc.y = fmaf(c, bj.y, acc.y);
                acc.z = fmaf(c, bj.z, acc.z);
                acc.w = fmaf(c, bj.w, acc.w);
            }
            acc.x = fmaf(fdec, hv[v].x, acc.x);
            acc.y = fmaf(fdec, hv[v].y, acc.y);
            acc.z = fmaf(fdec, hv[v].z, acc.z);
            acc.w = fmaf(fdec, hv[v].w, acc.w);
            if (a.ckpt_f16) {
                // stochastic rounding to FP16; acc becomes the rounded values (the read copy
                // below is built from the stored checkpoint)
                const uint2 w = sr_f16x4(acc, (uint32_t)col4, (uint32_t)(p0 + row), (uint32_t)h, (uint32_t)sb,
                                         a.seed_lo, a.seed_hi);
                __stcs(reinterpret_cast<uint2 *>(a.ckpt) + tile * N / 4 + tid + v * nthr, w);
            } else {
                st_stream(reinterpret_cast<float4 *>(a.ckpt + tile * N) + tid + v * nthr, acc);
            }
            if (a.read_copy == 2) {
                const float m4 = fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w)));
                const float m = group_max<G4>(m4), mb = group_max<4>(m4);
                float s_r, k_r, inv;
                nv4_row_scale(m, s_r, k_r);
                const uint32_t sbc = nv4_block_scale(mb, s_r, k_r, inv);
                uint8_t *hq = a.ckpt_q + ((size_t)sb * H + h) * nv4_head_bytes(P, N);
                const int prow = p0 + row;
                reinterpret_cast<uint16_t *>(hq + (size_t)prow * (N / 2))[col4] = (uint16_t)e2m1_pack4(
                    __fmul_rn(acc.x, inv), __fmul_rn(acc.y, inv), __fmul_rn(acc.z, inv), __fmul_rn(acc.w, inv));
                if ((col4 & 3) == 0) hq[P * N / 2 + prow * (N / 16) + col4 / 4] = (uint8_t)sbc;
                if (col4 == 0) a.ckpt_scale[tile + row] = s_r;
            } else if (a.read_copy) {
                float m = fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w)));
                m = group_max<G4>(m);
                float scale, inv;
                e4m3_row_scale(m, scale, inv);
                const uint32_t code = e4m3_pack4(__fmul_rn(acc.x, inv), __fmul_rn(acc.y, inv),
                                                 __fmul_rn(acc.z, inv), __fmul_rn(acc.w, inv));
                reinterpret_cast<uint32_t *>(a.ckpt_q + tile * N)[tid + v * nthr] = code;
                if (col4 == 0) a.ckpt_scale[tile + row] = scale;
            }
        }
    }
    if constexpr (TQ > 0) {
        float part[NQV * VPT];
#pragma unroll
        for (int i = 0; i < NQV; ++i) {
            float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < nq) c = *reinterpret_cast<const float4 *>(s_C + i * N + col4 * 4);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                float4 hh;
                float sc = 1.0f;
                if (use_q) { hh = a.read_copy == 2 ? e2m1_unpack4(qv[v]) : e4m3_unpack4(qv[v]); sc = qs[v]; }
                else hh = hv[v];
                float d = hh.x * c.x;
                d = fmaf(hh.y, c.y, d);
                d = fmaf(hh.z, c.z, d);
                d = fmaf(hh.w, c.w, d);
                part[i * VPT + v] = d * sc;
            }
        }
        group_reduce<G4, NQV * VPT>(part);
        if (reduced_writer<G4, NQV * VPT>()) {
            constexpr int NV = (NQV * VPT <= G4) ? 1 : (NQV * VPT) / G4;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = reduced_index<G4, NQV * VPT>(k);
                const int i = vi / VPT, v = vi - i * VPT;
                if (i < nq) s_yck[i * R + row0 + v * rstep] = part[k];
            }
        }
    }
    __syncthreads();

    // ---- 5. outputs, this CTA's x records
    if constexpr (TQ > 0) {
        for (int idx = tid; idx < nq * R; idx += nthr) {
            const int i = idx / R, r = idx - i * R;
            const float out = fmaf(s_decay[i], s_yck[idx], s_rt[idx]);
            const size_t yrow = MODE == kVerify ? (((size_t)b * a.T + i) * H + h) : ((size_t)b * H + h);
            a.y[yrow * P + p0 + r] = out;
        }
    }
    // new-record slots: decode appends at (head + len) unless it folded the
    // token; verify appends drafts after the (possibly just emptied) buffer
    const int head2 = (MODE == kVerify && fold) ? (head + len) % L : head;
    const int len2 = (MODE == kVerify && fold) ? 0 : len;
    const int nnew = MODE == kVerify ? a.T : ((MODE == kDecode && !fold) ? 1 : 0);
    {
        char *wx_ = static_cast<char *>(a.rec_x);
        for (int idx = tid; idx < nnew * cx; idx += nthr) {
            const int i = idx / cx, c = idx - i * cx;
            const int slot = (head2 + len2 + i) % L;
            const size_t irow = MODE == kVerify ? (((size_t)b * a.T + i) * H + h) : ((size_t)b * H + h);
            const uint4 val = __ldcg(reinterpret_cast<const uint4 *>(ix + (irow * P + p0 + c * E) * esz));
            *reinterpret_cast<uint4 *>(wx_ + ((((size_t)sb * H + h) * L + slot) * P + p0 + c * E) * esz) = val;
        }
    }

    // ---- 6. arrive; the last CTA of the sequence writes the shared records
    //         and commits the ring pointers
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(a.arrive + sb, 1);
        s_flag[0] = (prev == (int)gridDim.x - 1);
    }
    __syncthreads();
    if (!s_flag[0]) return;
    __threadfence();
    if (nnew > 0) {
        for (int idx = tid; idx < nnew * H; idx += nthr) {
            const int i = idx / H, hh = idx - i * H;
            const int slot = (head2 + len2 + i) % L;
            const float d = MODE == kVerify ? __ldcg(a.dt + ((size_t)b * a.T + i) * H + hh)
                                            : __ldcg(a.dt + (size_t)b * H + hh);
            a.rec_dt[((size_t)sb * H + hh) * L + slot] = d;
        }
        const int nBC = nnew * a.G * cB;
        char *wB = static_cast<char *>(a.rec_B);
        char *wC = static_cast<char *>(a.rec_C);
        for (int idx = tid; idx < 2 * nBC; idx += nthr) {
            const bool isC = idx >= nBC;
            if (isC && wC == nullptr) continue;
            const int k = isC ? idx - nBC : idx;
            const int i = k / (a.G * cB);
            const int r2 = k - i * a.G * cB;
            const int gg = r2 / cB, c = r2 - gg * cB;
            const int slot = (head2 + len2 + i) % L;
            const size_t irow = MODE == kVerify ? (((size_t)b * a.T + i) * a.G + gg) : ((size_t)b * a.G + gg);
            const char *src = (isC ? iC : iB) + (irow * N + c * E) * esz;
            char *dst = (isC ? wC : wB) + ((((size_t)sb * a.G + gg) * L + slot) * N + c * E) * esz;
            *reinterpret_cast<uint4 *>(dst) = __ldcg(reinterpret_cast<const uint4 *>(src));
        }
    }
    if (tid == 0) {
        int nh, nl;
        if (MODE == kDecode) {
            nh = fold ? (head + len + 1) % L : head;
            nl = fold ? 0 : len + 1;
        } else if (MODE == kVerify) {
            nh = head2;
            nl = len2 + a.T;
        } else {
            nh = (head + len) % L;
            nl = 0;
        }
        a.ring_head[sb] = nh;
        a.ring_len[sb] = nl;
        a.arrive[sb] = 0;
    }
}

}  // namespace rssm
