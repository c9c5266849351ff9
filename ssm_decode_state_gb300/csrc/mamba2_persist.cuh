// Persistent, TMA-pipelined Mamba-2 replay decode (the serving-shape path).
//
// One CTA per SM walks a static list of work items; an item is HPI heads of
// one group of one sequence.  The checkpoint of each head (P x N floats, or
// its FP8 read copy on non-flush steps) streams through an S-stage ring of
// shared-memory buffers filled by one-dimensional bulk copies (the TMA
// engine, `cp.async.bulk`) that complete on per-stage mbarriers; thread 0
// keeps S head tiles in flight ahead of the consumer, across item boundaries,
// so HBM never waits for the per-item bookkeeping.  The records an item needs
// (x of its heads, dt, the group's B, the current C) are prefetched one item
// ahead with cp.async into a double buffer.
//
// Per item: B_j . C_t for the group, decay weights per head, the record term
// per row; per head tile: row dot products with C_t (lanes of a row reduce
// with shuffles), y = exp(A S) (h_c . C_t) + record term; on flush steps the
// fold h_c <- exp(A S) h_c + sum_j w_j x_j B_j^T is written back (and the FP8
// copy re-quantised).  The CTA that sees the last arrival of a sequence
// commits its ring pointers.
#pragma once

#include "mamba2_replay.cuh"

namespace rssm {

struct PersistCfg {
    int items;     // B * H / HPI
    int nchunk;    // head chunks per group = hpg / HPI
    int stages;    // S
    int arrivals;  // items per sequence = H / HPI
};

// Byte layout of the persistent kernel's shared memory.
struct PSmem {
    int stage_bytes, stages_off, mbar_off;
    int rec_off[2], rx_off, rB_off, rC_off, rdt_off, rec_bytes;
    int cb_off, w_off, decay_off, rt_off, yck_off, wx_off, meta_off, flag_off, total;
    __host__ __device__ PSmem(int P, int N, int L, int HPI, int S) {
        const int KM = L + 1;
        auto up = [](int v, int a) { return (v + a - 1) / a * a; };
        stage_bytes = P * N * 4;
        int o = 0;
        stages_off = o; o += S * stage_bytes;
        mbar_off = o;   o += up(S * 8, 16);
        // one record buffer: x [HPI][KM][P] bf16, B [KM][N] bf16, C [N] bf16, dt [HPI][KM] f32
        rx_off = 0;
        rB_off = up(HPI * KM * P * 2, 16);
        rC_off = rB_off + up(KM * N * 2, 16);
        rdt_off = rC_off + up(N * 2, 16);
        rec_bytes = up(rdt_off + HPI * KM * 4, 128);
        rec_off[0] = o; o += rec_bytes;
        rec_off[1] = o; o += rec_bytes;
        cb_off = o;    o += up(KM * 4, 16);
        w_off = o;     o += up(HPI * KM * 4, 16);
        decay_off = o; o += up(HPI * 4, 16);
        rt_off = o;    o += up(HPI * P * 4, 16);
        yck_off = o;   o += up(P * 4, 16);
        wx_off = o;    o += up(KM * P * 4, 16);
        meta_off = o;  o += 64;
        flag_off = o;  o += 16;
        total = o;
    }
};

__device__ __forceinline__ float bf16_at(const uint16_t *p, int i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}

template <int N, int VPT, int HPI>
__global__ void __launch_bounds__(256, 1) m2_decode_persistent(const M2Args a, const PersistCfg pc) {
    constexpr int NT = 256;
    constexpr int G4 = N / 4;
    constexpr int P = NT * VPT * 4 / N;         // rows per head tile
    constexpr int ROWS_PER_V = NT / G4;         // rows between a thread's consecutive float4s
    extern __shared__ __align__(128) unsigned char smraw[];
    const int tid = threadIdx.x;
    const int L = a.L, H = a.H, G = a.G, hpg = a.hpg;
    const int KM = L + 1;
    const PSmem lay(P, N, L, HPI, pc.stages);
    const int S = pc.stages;
    unsigned char *stages = smraw + lay.stages_off;
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smraw + lay.mbar_off);
    float *s_cb = reinterpret_cast<float *>(smraw + lay.cb_off);
    float *s_w = reinterpret_cast<float *>(smraw + lay.w_off);
    float *s_decay = reinterpret_cast<float *>(smraw + lay.decay_off);
    float *s_rt = reinterpret_cast<float *>(smraw + lay.rt_off);
    float *s_yck = reinterpret_cast<float *>(smraw + lay.yck_off);
    float *s_wx = reinterpret_cast<float *>(smraw + lay.wx_off);
    int *s_meta = reinterpret_cast<int *>(smraw + lay.meta_off);   // [MQ items][head, len]
    int *s_flag = reinterpret_cast<int *>(smraw + lay.flag_off);

    const int grid = gridDim.x;
    const int n_my = (pc.items - (int)blockIdx.x + grid - 1) / grid;
    if (n_my <= 0) return;
    const int n_tiles = n_my * HPI;
    const bool q8 = a.read_copy != 0;
    const uint64_t pol = l2_evict_first_policy();

    auto item_of = [&](int k) { return (int)blockIdx.x + k * grid; };
    // item -> (b, g, c): item = (b * G + g) * nchunk + c
    auto item_b = [&](int it) { return it / (G * pc.nchunk); };
    auto item_h0 = [&](int it) {
        const int bg = it / pc.nchunk, c = it - bg * pc.nchunk;
        return (bg % G) * hpg + c * HPI;
    };

    // ---- thread 0: ring pointers.  Each item's pointers are read exactly once
    // (by whichever of the producer or the consumer needs them first) into a
    // small ring in shared memory, and the item arrives on its sequence's
    // counter right after the read; the returned count is checked at the next
    // arrival, and the CTA that saw the last arrival commits the new pointers.
    // No item can see a committed value: the commit needs its own arrival.
    constexpr int MQ = 8;
    int loaded = -1;
    int pend_b = -1, pend_prev = 0, pend_head = 0, pend_len = 0;
    auto resolve = [&]() {
        if (pend_b < 0) return;
        if (pend_prev == pc.arrivals - 1) {
            __threadfence();
            const bool bad = pend_head < 0 || pend_head >= L || pend_len < 0 || pend_len > L;
            if (!bad) {
                const bool fold = pend_len + 1 >= L;
                a.ring_head[pend_b] = fold ? (pend_head + pend_len + 1) % L : pend_head;
                a.ring_len[pend_b] = fold ? 0 : pend_len + 1;
            }
            a.arrive[pend_b] = 0;
        }
        pend_b = -1;
    };
    auto meta_of = [&](int k) {                   // thread 0 only
        while (loaded < k) {
            ++loaded;
            const int it = item_of(loaded);
            const int b = item_b(it);
            const int hd = __ldcg(a.ring_head + b), ln = __ldcg(a.ring_len + b);
            s_meta[(loaded % MQ) * 2 + 0] = hd;
            s_meta[(loaded % MQ) * 2 + 1] = ln;
            resolve();
            __threadfence();
            pend_prev = atomicAdd(a.arrive + b, 1);
            pend_b = b; pend_head = hd; pend_len = ln;
            if ((hd < 0 || hd >= L || ln < 0 || ln > L) && item_h0(it) == 0) flag_error(a.err, RSSM_DEVERR_RING_META);
        }
    };

    // ---- thread 0: the producer; tile t goes to stage t % S
    auto issue = [&](int t) {
        const int k = t / HPI, hh = t - k * HPI;
        const int it = item_of(k);
        const int b = item_b(it), h = item_h0(it) + hh;
        meta_of(k);
        const int ln = s_meta[(k % MQ) * 2 + 1], hd = s_meta[(k % MQ) * 2 + 0];
        const bool fold_or_bad = (ln + 1 >= L) || ln < 0 || ln > L || hd < 0 || hd >= L;
        uint64_t *bar = mbar + (t % S);
        unsigned char *dst = stages + (t % S) * lay.stage_bytes;
        const size_t tile = ((size_t)b * H + h) * P;
        if (q8 && !fold_or_bad) {
            mbar_arrive_expect_tx(bar, P * N + P * 4);
            bulk_g2s(dst, a.ckpt_q + tile * N, P * N, bar, pol);
            bulk_g2s(dst + P * N, a.ckpt_scale + tile, P * 4, bar, pol);
        } else {
            mbar_arrive_expect_tx(bar, P * N * 4);
            bulk_g2s(dst, a.ckpt + tile * N, P * N * 4, bar, pol);
        }
    };

    // ---- records of item k -> record buffer k & 1 (all threads, cp.async)
    auto prefetch_records = [&](int k) {
        const int it = item_of(k);
        const int b = item_b(it), h0 = item_h0(it), g = h0 / hpg;
        const int hd = s_meta[(k % MQ) * 2 + 0], ln = s_meta[(k % MQ) * 2 + 1];
        if (hd < 0 || hd >= L || ln < 0 || ln > L) return;
        const int nrec = ln + 1;
        unsigned char *rb = smraw + lay.rec_off[k & 1];
        const uint16_t *rx = static_cast<const uint16_t *>(a.rec_x);
        const uint16_t *rB = static_cast<const uint16_t *>(a.rec_B);
        const uint16_t *ix = static_cast<const uint16_t *>(a.x);
        const uint16_t *iB = static_cast<const uint16_t *>(a.Bin);
        const uint16_t *iC = static_cast<const uint16_t *>(a.Cin);
        constexpr int CX = P / 8, CB = N / 8;
        const int nx = HPI * nrec * CX, nB = nrec * CB, nC = CB, ndt = HPI * nrec;
        const int total = nx + nB + nC + ndt;
        for (int idx = tid; idx < total; idx += NT) {
            if (idx < nx) {
                const int hh = idx / (nrec * CX);
                const int r = idx - hh * nrec * CX;
                const int j = r / CX, c = r - j * CX;
                const size_t bh = (size_t)b * H + h0 + hh;
                const uint16_t *src = j < ln ? rx + ((bh * L + (hd + j) % L) * P + c * 8) : ix + (bh * P + c * 8);
                cp_async16(rb + lay.rx_off + ((hh * KM + j) * P + c * 8) * 2, src);
            } else if (idx < nx + nB) {
                const int r = idx - nx;
                const int j = r / CB, c = r - j * CB;
                const uint16_t *src = j < ln ? rB + ((((size_t)b * G + g) * L + (hd + j) % L) * N + c * 8)
                                             : iB + (((size_t)b * G + g) * N + c * 8);
                cp_async16(rb + lay.rB_off + (j * N + c * 8) * 2, src);
            } else if (idx < nx + nB + nC) {
                const int c = idx - nx - nB;
                cp_async16(rb + lay.rC_off + c * 16, iC + (((size_t)b * G + g) * N + c * 8));
            } else {
                const int r = idx - nx - nB - nC;
                const int hh = r / nrec, j = r - hh * nrec;
                const size_t bh = (size_t)b * H + h0 + hh;
                const float *src = j < ln ? a.rec_dt + bh * L + (hd + j) % L : a.dt + bh;
                cp_async4(rb + lay.rdt_off + (hh * KM + j) * 4, src);
            }
        }
        cp_async_commit();
    };

    // ---- prologue
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(mbar + s, 1);
        fence_mbar_init();
        s_flag[0] = 0;
        meta_of(0);
    }
    __syncthreads();
    if (tid == 0) {
        for (int t = 0; t < S && t < n_tiles; ++t) issue(t);
    }
    prefetch_records(0);

    const int col4 = tid % G4;
    const int row0 = tid / G4;

    for (int k = 0; k < n_my; ++k) {
        const int it = item_of(k);
        const int b = item_b(it), h0 = item_h0(it), g = h0 / hpg;
        cp_async_wait_all();
        __syncthreads();                                      // records of item k landed
        const int hd = s_meta[(k % MQ) * 2 + 0], ln = s_meta[(k % MQ) * 2 + 1];
        const bool bad = hd < 0 || hd >= L || ln < 0 || ln > L;
        const bool fold = !bad && (ln + 1 >= L);
        const int nrec = ln + 1;
        const unsigned char *rb = smraw + lay.rec_off[k & 1];
        const uint16_t *r_x = reinterpret_cast<const uint16_t *>(rb + lay.rx_off);
        const uint16_t *r_B = reinterpret_cast<const uint16_t *>(rb + lay.rB_off);
        const uint16_t *r_C = reinterpret_cast<const uint16_t *>(rb + lay.rC_off);
        const float *r_dt = reinterpret_cast<const float *>(rb + lay.rdt_off);
        if (tid == 0 && k + 1 < n_my) meta_of(k + 1);
        if (!bad) {
            // B_j . C_t, one warp per record
            const int warp = tid >> 5, lane = tid & 31;
            for (int j = warp; j < nrec; j += NT / 32) {
                float acc = 0.0f;
                for (int n = lane; n < N; n += 32) acc = fmaf(bf16_at(r_B, j * N + n), bf16_at(r_C, n), acc);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (lane == 0) s_cb[j] = acc;
            }
            // decay weights per head: w_j = exp(A sum(dt after j)) dt_j, and exp(A S)
            for (int idx = tid; idx < HPI * KM; idx += NT) {
                const int hh = idx / KM, j = idx - hh * KM;
                const float Ah = a.A[h0 + hh];
                const float *dth = r_dt + hh * KM;
                if (j < nrec) s_w[idx] = expf(Ah * suffix_sum(dth, j, ln)) * dth[j];
            }
            for (int hh = tid; hh < HPI; hh += NT)
                s_decay[hh] = expf(a.A[h0 + hh] * suffix_sum(r_dt + hh * KM, -1, ln));
        }
        __syncthreads();                                      // cb, w, decay; next meta
        if (!bad) {
            for (int idx = tid; idx < HPI * P; idx += NT) {
                const int hh = idx / P, p = idx - hh * P;
                const float *wh = s_w + hh * KM;
                const uint16_t *xh = r_x + hh * KM * P;
                float acc = 0.0f;
                for (int j = 0; j < nrec; ++j) acc = fmaf(wh[j] * s_cb[j], bf16_at(xh, j * P + p), acc);
                s_rt[idx] = fmaf(a.D[h0 + hh], bf16_at(xh, ln * P + p), acc);
            }
        }
        if (k + 1 < n_my) prefetch_records(k + 1);
        __syncthreads();                                      // rt ready

        // C_t fragment of this lane's 4 columns
        float4 cfr = make_float4(bf16_at(r_C, col4 * 4 + 0), bf16_at(r_C, col4 * 4 + 1),
                                 bf16_at(r_C, col4 * 4 + 2), bf16_at(r_C, col4 * 4 + 3));
        for (int hh = 0; hh < HPI; ++hh) {
            const int t = k * HPI + hh;
            const int st = t % S;
            const bool ok = mbar_wait(mbar + st, (uint32_t)((t / S) & 1));
            if (!ok) s_flag[0] = 1;
            const unsigned char *stg = stages + st * lay.stage_bytes;
            float4 hv[VPT];
            const bool use_q = q8 && !fold && !bad;
            if (use_q) {
                const uint32_t *q = reinterpret_cast<const uint32_t *>(stg);
                const float *sc = reinterpret_cast<const float *>(stg + P * N);
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const float4 d = e4m3_unpack4(q[tid + v * NT]);
                    const float s = sc[row0 + v * ROWS_PER_V];
                    hv[v] = make_float4(d.x * s, d.y * s, d.z * s, d.w * s);
                }
            } else {
#pragma unroll
                for (int v = 0; v < VPT; ++v) hv[v] = reinterpret_cast<const float4 *>(stg)[tid + v * NT];
            }
            if (fold) {
                const float *wh = s_w + hh * KM;
                const uint16_t *xh = r_x + hh * KM * P;
                for (int idx = tid; idx < nrec * P; idx += NT) {
                    const int j = idx / P;
                    s_wx[idx] = wh[j] * bf16_at(xh, idx);
                }
            }
            __syncthreads();                                  // stage consumed; wx ready
            if (s_flag[0]) {
                // a copy never completed: record it, stop issuing, drain what is in flight
                if (tid == 0) {
                    flag_error(a.err, RSSM_DEVERR_TIMEOUT);
                    for (int u = t + 1; u < t + S && u < n_tiles; ++u) mbar_wait(mbar + (u % S), (uint32_t)((u / S) & 1));
                }
                return;
            }
            if (tid == 0 && t + S < n_tiles) issue(t + S);
            if (!bad) {
                const int h = h0 + hh;
                float part[VPT];
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    float d = hv[v].x * cfr.x;
                    d = fmaf(hv[v].y, cfr.y, d);
                    d = fmaf(hv[v].z, cfr.z, d);
                    d = fmaf(hv[v].w, cfr.w, d);
                    part[v] = d;
                }
                group_reduce<G4, VPT>(part);
                if (reduced_writer<G4, VPT>()) {
                    constexpr int NV = (VPT <= G4) ? 1 : VPT / G4;
#pragma unroll
                    for (int kk = 0; kk < NV; ++kk) s_yck[row0 + reduced_index<G4, VPT>(kk) * ROWS_PER_V] = part[kk];
                }
                if (fold) {
                    const float dec = s_decay[hh];
                    const size_t tile = ((size_t)b * H + h) * P;
                    float4 *ckp = reinterpret_cast<float4 *>(a.ckpt + tile * N);
#pragma unroll
                    for (int v = 0; v < VPT; ++v) {
                        const int row = row0 + v * ROWS_PER_V;
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int j = 0; j < nrec; ++j) {
                            const float c = s_wx[j * P + row];
                            const uint2 braw = *reinterpret_cast<const uint2 *>(r_B + j * N + col4 * 4);
                            acc.x = fmaf(c, bf16lo(braw.x), acc.x);
                            acc.y = fmaf(c, bf16hi(braw.x), acc.y);
                            acc.z = fmaf(c, bf16lo(braw.y), acc.z);
                            acc.w = fmaf(c, bf16hi(braw.y), acc.w);
                        }
                        acc.x = fmaf(dec, hv[v].x, acc.x);
                        acc.y = fmaf(dec, hv[v].y, acc.y);
                        acc.z = fmaf(dec, hv[v].z, acc.z);
                        acc.w = fmaf(dec, hv[v].w, acc.w);
                        st_stream(ckp + tid + v * NT, acc);
                        if (q8) {
                            float m = fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w)));
                            m = group_max<G4>(m);
                            float scale, inv;
                            e4m3_row_scale(m, scale, inv);
                            reinterpret_cast<uint32_t *>(a.ckpt_q + tile * N)[tid + v * NT] =
                                e4m3_pack4(__fmul_rn(acc.x, inv), __fmul_rn(acc.y, inv), __fmul_rn(acc.z, inv),
                                           __fmul_rn(acc.w, inv));
                            if (col4 == 0) a.ckpt_scale[tile + row] = scale;
                        }
                    }
                }
            }
            __syncthreads();                                  // yck ready
            if (!bad && tid < P) {
                const int h = h0 + hh;
                a.y[((size_t)b * H + h) * P + tid] = fmaf(s_decay[hh], s_yck[tid], s_rt[hh * P + tid]);
            }
        }
        // ---- new records of this item (a non-flush step appends the token)
        if (!bad && !fold) {
            const int slot = (hd + ln) % L;
            constexpr int CX = P / 8, CB = N / 8;
            const uint16_t *ix = static_cast<const uint16_t *>(a.x);
            uint16_t *wx_ = static_cast<uint16_t *>(a.rec_x);
            const int nB = (h0 % hpg == 0) ? 2 * CB : 0;     // first chunk of the group writes B and C
            const int total = HPI * CX + nB + HPI;
            for (int idx = tid; idx < total; idx += NT) {
                if (idx < HPI * CX) {
                    const int hh = idx / CX, c = idx - hh * CX;
                    const size_t bh = (size_t)b * H + h0 + hh;
                    *reinterpret_cast<uint4 *>(wx_ + (bh * L + slot) * P + c * 8) =
                        __ldcg(reinterpret_cast<const uint4 *>(ix + bh * P + c * 8));
                } else if (idx < HPI * CX + nB) {
                    const int r = idx - HPI * CX;
                    const bool isC = r >= CB;
                    const int c = isC ? r - CB : r;
                    uint16_t *dst = static_cast<uint16_t *>(isC ? a.rec_C : a.rec_B);
                    if (dst == nullptr) continue;
                    const uint16_t *src = static_cast<const uint16_t *>(isC ? a.Cin : a.Bin);
                    *reinterpret_cast<uint4 *>(dst + ((((size_t)b * G + g) * L + slot) * N + c * 8)) =
                        __ldcg(reinterpret_cast<const uint4 *>(src + (((size_t)b * G + g) * N + c * 8)));
                } else {
                    const int hh = idx - HPI * CX - nB;
                    const size_t bh = (size_t)b * H + h0 + hh;
                    a.rec_dt[bh * L + slot] = __ldcg(a.dt + bh);
                }
            }
        }
    }
    if (tid == 0) resolve();
}

}  // namespace rssm
