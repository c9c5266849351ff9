// Persistent, warp-specialised replay decode of the gated delta rule at the
// serving head shape (dk = dv = 128, bf16 token inputs), with the fused flush.
//
// One CTA per SM walks a static list of work items, one (sequence, head)
// each; its dv x dk FP32 state streams through shared memory as two stages
// of 64 rows.  The ring pointers of every item are read (and committed by the
// last reader of each sequence) at kernel start; after that:
//
//  * tile warp (warp 0, one lane): bulk copies (TMA engine) of the state,
//    one 64-row half per stage, into an S-stage ring.
//  * record warp (warp 1): per item, the used ring slots of k and v (at most
//    two contiguous runs each) and the token's q, k, v by bulk copy, alpha
//    and beta by cp.async, into a ring of RB record buffers.
//  * preparation warps (two, after the consumers), alternate items, ahead of
//    the consumers: append the token to the ring; run the backward chain
//    u = q, d_j = k_j . u, u <- alpha_j (u - beta_j d_j k_j) (newest record
//    first), which leaves u_0 and the record term sum_j beta_j d_j v_j[r] of
//    every row, into item buffers handed over through mbarriers.
//  * consumer warps (eight): per stage, each warp reads its own 8 rows, frees
//    the stage, reduces the row dot products with u_0 across its lanes and
//    writes o[r] = S_c[r] . u_0 + record term; on the flush step it folds the
//    records into its rows (the rank-one updates s <- alpha_j s + beta_j
//    (v_j[r] - alpha_j (s . k_j)) k_j, oldest first, re-associated through the
//    records' Gram matrix, which the preparation warps supply) and stores them.
//
// Every wait is bounded (~2 s, then RSSM_DEVERR_TIMEOUT and an orderly exit).
#pragma once

#include "persist_common.cuh"

namespace rssm {

struct GPArgs {
    int H, L, items, max_my, stages, recbufs;
    float *ckpt;
    uint16_t *rec_k, *rec_v;
    float *rec_alpha, *rec_beta;
    int32_t *ring_head, *ring_len, *arrive;
    uint32_t *err;
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    float *o;
    const int32_t *slots;   // [batch] cache slot of each batch row; nullptr: row b uses slot b
    int cap;                // sequences the cache arrays hold
    int T;                  // drafts per sequence (verify only)
    int skip_folds;         // decode: the items whose sequence folds this step go to the
                            // tensor-core fold phase; 0: the decode phase folds them itself
};

constexpr int kGdnRows = 64;     // state rows per stage
constexpr int kGdnBufs = 4;      // prepared-item buffers
constexpr int kGdnMaxL = 16;     // largest ring the persistent kernels take
constexpr int kGdnMaxRec = 20;   // records a fold may take: L + 1 (a decode after a verify filled
                                 // the ring folds L buffered records and its token), in fours
// fold constants of a prepared item: C [16][16], a [16], g [16], A (floats)
constexpr int kFcA = kGdnMaxRec * kGdnMaxRec, kFcG = kFcA + kGdnMaxRec, kFcT = kFcG + kGdnMaxRec;
constexpr int kFcStride = kFcT + 4;

// Byte layout of the decode phase's shared memory (the per-item ring pointers
// and item lists live after it, in the step kernel's common region).
struct GPSmem {
    int stage_bytes, stages_off, full_off, empty_off, rfull_off, rempty_off, pfull_off, pempty_off;
    int rk_off, rv_off, rq_off, ral_off, rbe_off, rec_bytes, rec_off;
    int u_off, rt_off, fc_off, f_off, flag_off, total;
    __host__ __device__ GPSmem(int DK, int DV, int L, int S, int RB) {
        const int KM = L + 1;
        auto up = [](int v, int a) { return (v + a - 1) / a * a; };
        stage_bytes = kGdnRows * DK * 4;
        int o = 0;
        stages_off = o; o += S * stage_bytes;
        full_off = o;   o += 8 * S;
        empty_off = o;  o += 8 * S;
        rfull_off = o;  o += 8 * RB;
        rempty_off = o; o += 8 * RB;
        pfull_off = o;  o += 8 * kGdnBufs;
        pempty_off = o; o += 8 * kGdnBufs;
        o = up(o, 128);
        // one record buffer: k [KM][DK] bf16, v [KM][DV] bf16, q [DK] bf16, alpha, beta [KM] f32
        rk_off = 0;
        rv_off = up(KM * DK * 2, 16);
        rq_off = rv_off + up(KM * DV * 2, 16);
        ral_off = rq_off + up(DK * 2, 16);
        rbe_off = ral_off + up(KM * 4, 16);
        rec_bytes = up(rbe_off + KM * 4, 128);
        rec_off = o;  o += RB * rec_bytes;
        u_off = o;    o += up(kGdnBufs * DK * 4, 16);       // u_0 per prepared item
        rt_off = o;   o += up(kGdnBufs * DV * 4, 16);       // record term per prepared item
        fc_off = o;   o += up(kGdnBufs * kFcStride * 4, 16); // fold constants per prepared item
        f_off = o;    o += up(8 * kGdnMaxRec * 8 * 4, 16);  // fold coefficients, [warp][j][8 rows]
        flag_off = o; o += 16;                              // abort flag
        total = o;
    }
};

// Fold constants of nr records (the preparation warps' share of a fold): the
// Gram entries C_ij = (k_i . k_j) prod_{i<m<j} alpha_m (i < j), the prefix
// products a_j = prod_{m<j} alpha_m, the suffix products g_j = prod_{m>j}
// alpha_m and the total product A, into fc (one warp, nr <= kGdnMaxRec).  The
// alphas travel in registers (lane m holds alpha_m); every product of alphas
// is taken in increasing m.
template <int DK>
__device__ __forceinline__ void gdn_fold_constants(float *fc, const uint16_t *r_k, const float *r_al, int nr) {
    constexpr int CK = DK / 8;                           // 16-byte chunks per k row
    const int lane = threadIdx.x & 31;
    const float al = lane < nr ? r_al[lane] : 1.0f;
    // the pairs i < j, one per lane and pass, numbered j (j - 1) / 2 + i: a dot product
    // of two bf16 rows (bf16-pair FMAs in two chains), times the alphas between them;
    // lanes start on different 16-byte chunks of their rows
    const int npairs = nr * (nr - 1) / 2;
    for (int p0 = 0; p0 < npairs; p0 += 32) {
        const int pidx = p0 + lane;
        const bool on = pidx < npairs;
        int j = 1;
        while ((j + 1) * j / 2 <= pidx) ++j;
        const int i = pidx - j * (j - 1) / 2;
        float t0 = 0.0f, t1 = 0.0f;
        if (on) {
            for (int cc = 0; cc < CK; ++cc) {
                const int c = (cc + lane) % CK;
                const uint4 ki = *reinterpret_cast<const uint4 *>(r_k + i * DK + c * 8);
                const uint4 kj = *reinterpret_cast<const uint4 *>(r_k + j * DK + c * 8);
                t0 = fma_bf16_pair(ki.x, kj.x, t0);
                t1 = fma_bf16_pair(ki.y, kj.y, t1);
                t0 = fma_bf16_pair(ki.z, kj.z, t0);
                t1 = fma_bf16_pair(ki.w, kj.w, t1);
            }
        }
        float pa = 1.0f;
        for (int m = 0; m < nr; ++m) {
            const float am = __shfl_sync(0xffffffffu, al, m);
            if (m > i && m < j) pa *= am;
        }
        if (on) fc[i * kGdnMaxRec + j] = (t0 + t1) * pa;
    }
    float pre = 1.0f, suf = 1.0f, tot = 1.0f;
    for (int m = 0; m < nr; ++m) {
        const float am = __shfl_sync(0xffffffffu, al, m);
        if (m < lane) pre *= am;
        if (m > lane) suf *= am;
        tot *= am;
    }
    if (lane < nr) {
        fc[kFcA + lane] = pre;
        fc[kFcG + lane] = suf;
    }
    if (lane == 0) fc[kFcT] = tot;
}

// A consumer warp's share of a fold: its 8 rows cw + 8 v (v < VPT) of stage uu,
// held in hv, take the nrec records' rank-one updates s <- alpha_j s + beta_j
// (v_j[r] - alpha_j (s . k_j)) k_j, oldest first, re-associated: with p_j =
// s_c . k_j, d_j = s_j . k_j = a_j p_j + sum_{i<j} C_ij e_i and e_j = beta_j
// (v_j[r] - alpha_j d_j), the folded row is A s_c + sum_j e_j g_j k_j (fc holds
// C, a, g, A).  Rows no longer wait on one another's reductions record by
// record; the state is rounded once.  The rows are stored to ck4 (the stage's
// first row in the cache); sf is the warp's [16][8] scratch.
template <int DK, int DV, int VPT>
__device__ __forceinline__ void gdn_fold_stage(float4 (&hv)[VPT], int nrec, const uint16_t *r_k, const uint16_t *r_v,
                                               const float *r_al, const float *r_be, const float *fc, float *sf,
                                               int uu, int cw, float4 *ck4) {
    constexpr int NC = 256, RSTEP = NC / (DK / 4);
    const int lane = threadIdx.x & 31, col4 = lane, ctid = cw * 32 + lane;
    // projections of the warp's 8 rows, 4 records at a time; after the
    // reduction lane l holds row l / 4, record 4 q + l % 4
    constexpr int NQ = kGdnMaxRec / 4;
    float pq[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        pq[q] = 0.0f;
        if (4 * q >= nrec) continue;                     // warp-uniform
        float t[VPT * 4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = q * 4 + jj;
            float4 kj = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < nrec) {
                const uint2 kraw = *reinterpret_cast<const uint2 *>(r_k + j * DK + col4 * 4);
                kj = make_float4(bf16lo(kraw.x), bf16hi(kraw.x), bf16lo(kraw.y), bf16hi(kraw.y));
            }
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                float d = hv[v].x * kj.x;
                d = fmaf(hv[v].y, kj.y, d);
                d = fmaf(hv[v].z, kj.z, d);
                d = fmaf(hv[v].w, kj.w, d);
                t[v * 4 + jj] = d;
            }
        }
        group_reduce<32, VPT * 4>(t);
        pq[q] = t[0];
    }
    // each lane of a quad gathers its row's projections and runs the recurrence
    float p[kGdnMaxRec];
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
        for (int src = 0; src < 4; ++src) p[q * 4 + src] = __shfl_sync(0xffffffffu, pq[q], (lane & ~3) + src);
    const int vrow = lane >> 2, row = uu * kGdnRows + cw + RSTEP * vrow;
    float acc[kGdnMaxRec], f[kGdnMaxRec];
#pragma unroll
    for (int m = 0; m < kGdnMaxRec; ++m) acc[m] = 0.0f;
#pragma unroll
    for (int j = 0; j < kGdnMaxRec; ++j) {
        f[j] = 0.0f;
        if (j < nrec) {
            const float dj = fmaf(fc[kFcA + j], p[j], acc[j]);
            const float ej = r_be[j] * fmaf(-r_al[j], dj, bf16_at(r_v, j * DV + row));
            f[j] = ej * fc[kFcG + j];
#pragma unroll
            for (int m = j + 1; m < kGdnMaxRec; ++m) acc[m] = fmaf(fc[j * kGdnMaxRec + m], ej, acc[m]);
        }
    }
    if ((lane & 3) == 0) {
#pragma unroll
        for (int j = 0; j < kGdnMaxRec; ++j) sf[j * 8 + vrow] = f[j];
    }
    __syncwarp();
    // rank-nrec update, then the decayed state in one fma
    unsigned long long acc01[VPT], acc23[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) acc01[v] = acc23[v] = 0ull;
    for (int j = 0; j < nrec; ++j) {
        const uint2 kraw = *reinterpret_cast<const uint2 *>(r_k + j * DK + col4 * 4);
        const unsigned long long b01 = f2pack(bf16lo(kraw.x), bf16hi(kraw.x));
        const unsigned long long b23 = f2pack(bf16lo(kraw.y), bf16hi(kraw.y));
        const float4 fa = *reinterpret_cast<const float4 *>(sf + j * 8);
        const float4 fb = *reinterpret_cast<const float4 *>(sf + j * 8 + 4);
        const float fv[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const unsigned long long cc = f2pack(fv[v], fv[v]);
            acc01[v] = fma2(cc, b01, acc01[v]);
            acc23[v] = fma2(cc, b23, acc23[v]);
        }
    }
    const unsigned long long tt = f2pack(fc[kFcT], fc[kFcT]);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        float4 o;
        f2unpack(fma2(tt, f2pack(hv[v].x, hv[v].y), acc01[v]), o.x, o.y);
        f2unpack(fma2(tt, f2pack(hv[v].z, hv[v].w), acc23[v]), o.z, o.w);
        st_stream(ck4 + ctid + v * NC, o);
    }
    __syncwarp();                                        // sf is rewritten by the next stage
}

// The decode phase of a step (see gdn_decode_persistent): the n_work items of
// s_list (indices into this CTA's static item list; s_meta holds their ring
// pointers as read at kernel start).  smraw is the 1024-byte aligned base of
// the dynamic shared memory.
template <int DK, int DV>
__device__ __forceinline__ void gdn_decode_phase(const GPArgs &a, unsigned char *smraw, const int *s_meta,
                                                 const int *s_list, int n_work) {
    constexpr int NC = 256, VPT = 8, G4 = DK / 4, RSTEP = NC / G4, NU = DV / kGdnRows;
    static_assert(G4 == 32 && NC * VPT * 4 == kGdnRows * DK && DV % kGdnRows == 0, "serving shape");
    constexpr int CK = DK / 8, CV = DV / 8;              // 16-byte chunks per k / v row
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.L, H = a.H, S = a.stages, RB = a.recbufs;
    const GPSmem lay(DK, DV, L, S, RB);
    unsigned char *stages = smraw + lay.stages_off;
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + lay.full_off);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smraw + lay.empty_off);
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smraw + lay.rfull_off);
    uint64_t *rempty = reinterpret_cast<uint64_t *>(smraw + lay.rempty_off);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smraw + lay.pfull_off);
    uint64_t *pempty = reinterpret_cast<uint64_t *>(smraw + lay.pempty_off);
    float *s_u = reinterpret_cast<float *>(smraw + lay.u_off);
    float *s_rt = reinterpret_cast<float *>(smraw + lay.rt_off);
    float *s_fc = reinterpret_cast<float *>(smraw + lay.fc_off);
    float *s_f = reinterpret_cast<float *>(smraw + lay.f_off);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smraw + lay.flag_off);

    const int grid = gridDim.x;
    auto item_of = [&](int k) { return (int)blockIdx.x + k * grid; };   // item = b * H + h
    auto meta_bad = [&](int hd, int ln) { return hd < 0 || hd >= L || ln < 0 || ln > L; };
    auto rec = [&](int r) { return smraw + lay.rec_off + r * lay.rec_bytes; };
    // (cache slot, head) of item k: where its checkpoint and records live
    auto cb_of = [&](int k) { return (size_t)s_meta[k * 3 + 2] * H + (size_t)(item_of(k) % H); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, NC / 32);               // one arrival per consumer warp
        }
        for (int r = 0; r < RB; ++r) {
            mbar_init(rfull + r, 33);                    // 32 cp.async arrivals + lane 0's
            mbar_init(rempty + r, NC / 32);
        }
        for (int i = 0; i < kGdnBufs; ++i) {
            mbar_init(pfull + i, 1);                     // the preparing warp's lane 0
            mbar_init(pempty + i, NC / 32);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ================================= tile warp ==================================
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first_policy();
        bool ok = true;
        int issued = 0;
        for (int w = 0; w < n_work && ok; ++w) {
            const size_t cbh = cb_of(s_list[w]);             // cache
            for (int uu = 0; uu < NU; ++uu) {
                const int t = issued, s = t % S;
                if (t >= S) ok = pwait(empty + s, (uint32_t)(((t / S) - 1) & 1), s_abort) && !*s_abort;
                if (!ok) break;
                mbar_arrive_expect_tx(full + s, lay.stage_bytes);
                bulk_g2s(stages + s * lay.stage_bytes, a.ckpt + (cbh * DV + uu * kGdnRows) * DK, lay.stage_bytes,
                         full + s, pol);
                issued = t + 1;
            }
        }
        if (!ok) {
            // a wait gave up, or another warp did: tell everyone
            *s_abort = 1;
            flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        }
        // the copies in flight must land before the CTA ends.  Normally the
        // consumers waited for every one, but after an abort they stop waiting;
        // the stages of older units were refilled only after every consumer warp
        // waited for them (an aborted warp's release is seen above as the abort)
        for (int u = issued - S < 0 ? 0 : issued - S; u < issued; ++u)
            mbar_wait(full + (u % S), (uint32_t)((u / S) & 1));
        return;
    }

    if (warp == 1) {
        // ================================ record warp =================================
        bool ok = true;
        int w = 0;
        for (; w < n_work; ++w) {
            const int k = s_list[w], r = w % RB;
            if (lane == 0 && w >= RB) ok = pwait(rempty + r, (uint32_t)(((w / RB) - 1) & 1), s_abort) && !*s_abort;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const size_t bh = (size_t)item_of(k), cbh = cb_of(k);    // inputs, cache
            const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1];
            const bool good = !meta_bad(hd, ln);
            if (good) {
                // list position j < ln is ring slot (hd + j) mod L, j = ln the token
                unsigned char *rb = rec(r);
                const int nrec = ln + 1;
                const int run1 = ln < L - hd ? ln : L - hd, run2 = ln - run1;
                if (lane == 0) mbar_arrive_expect_tx(rfull + r, (uint32_t)((nrec * (DK + DV) + DK) * 2));
                __syncwarp();
                if (lane == 0) {
                    unsigned char *d = rb + lay.rk_off;
                    if (run1) bulk_g2s(d, a.rec_k + (cbh * L + hd) * DK, run1 * DK * 2, rfull + r);
                    if (run2) bulk_g2s(d + run1 * DK * 2, a.rec_k + cbh * L * DK, run2 * DK * 2, rfull + r);
                    bulk_g2s(d + ln * DK * 2, a.k + bh * DK, DK * 2, rfull + r);
                } else if (lane == 1) {
                    unsigned char *d = rb + lay.rv_off;
                    if (run1) bulk_g2s(d, a.rec_v + (cbh * L + hd) * DV, run1 * DV * 2, rfull + r);
                    if (run2) bulk_g2s(d + run1 * DV * 2, a.rec_v + cbh * L * DV, run2 * DV * 2, rfull + r);
                    bulk_g2s(d + ln * DV * 2, a.v + bh * DV, DV * 2, rfull + r);
                } else if (lane == 2) {
                    bulk_g2s(rb + lay.rq_off, a.q + bh * DK, DK * 2, rfull + r);
                }
                for (int j = lane; j <= ln; j += 32) {
                    const int slot = hd + j < L ? hd + j : hd + j - L;
                    cp_async4(rb + lay.ral_off + j * 4, j < ln ? a.rec_alpha + cbh * L + slot : a.alpha + bh);
                    cp_async4(rb + lay.rbe_off + j * 4, j < ln ? a.rec_beta + cbh * L + slot : a.beta + bh);
                }
            }
            cp_async_arrive_noinc(rfull + r);
            if (lane == 0 && !good) mbar_arrive(rfull + r);
        }
        cp_async_wait_all();
        // the copies of the last items may still be in flight: wait (bounded)
        if (lane == 0)
            for (int kk = w - RB < 0 ? 0 : w - RB; kk < w; ++kk) mbar_wait(rfull + kk % RB, (uint32_t)((kk / RB) & 1));
        if (!ok && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        }
        return;
    }

    if (warp >= 2 + NC / 32) {
        // ============================ item-preparation warps ============================
        const int pw = warp - 2 - NC / 32;               // 0 or 1: even or odd items
        bool live = true;
        for (int w = pw; w < n_work; w += 2) {
            const int kk = s_list[w], r = w % RB, ib = w % kGdnBufs;
            if (live && w >= kGdnBufs && !pwait(pempty + ib, (uint32_t)(((w / kGdnBufs) - 1) & 1), s_abort)) {
                live = false;
                *s_abort = 1;
            }
            if (live && !pwait(rfull + r, (uint32_t)((w / RB) & 1), s_abort)) {
                live = false;
                *s_abort = 1;
            }
            const size_t cbh = cb_of(kk);                    // the preparation writes the cache only
            const int hd = s_meta[kk * 3 + 0], ln = s_meta[kk * 3 + 1];
            const bool work = live && !meta_bad(hd, ln);
            const unsigned char *rb = rec(r);
            const uint16_t *r_k = reinterpret_cast<const uint16_t *>(rb + lay.rk_off);
            const uint16_t *r_v = reinterpret_cast<const uint16_t *>(rb + lay.rv_off);
            const uint16_t *r_q = reinterpret_cast<const uint16_t *>(rb + lay.rq_off);
            const float *r_al = reinterpret_cast<const float *>(rb + lay.ral_off);
            const float *r_be = reinterpret_cast<const float *>(rb + lay.rbe_off);
            if (work && ln + 1 < L) {
                // a non-flush step appends the token to the ring, slot (hd + ln) mod L
                const int slot = hd + ln < L ? hd + ln : hd + ln - L;
                if (lane < CK) {
                    *reinterpret_cast<uint4 *>(a.rec_k + (cbh * L + slot) * DK + lane * 8) =
                        *reinterpret_cast<const uint4 *>(r_k + ln * DK + lane * 8);
                } else if (lane < CK + CV) {
                    const int c = lane - CK;
                    *reinterpret_cast<uint4 *>(a.rec_v + (cbh * L + slot) * DV + c * 8) =
                        *reinterpret_cast<const uint4 *>(r_v + ln * DV + c * 8);
                }
                if (lane == 0) {
                    a.rec_alpha[cbh * L + slot] = r_al[ln];
                    a.rec_beta[cbh * L + slot] = r_be[ln];
                }
            }
            if (work) {
                // backward chain from the newest record; lane holds columns lane + 32 m of u
                // and rows lane + 32 m of the record term
                constexpr int MK = DK / 32, MV = DV / 32;
                float u[MK], racc[MV];
#pragma unroll
                for (int m = 0; m < MK; ++m) u[m] = bf16_at(r_q, lane + 32 * m);
#pragma unroll
                for (int m = 0; m < MV; ++m) racc[m] = 0.0f;
                for (int j = ln; j >= 0; --j) {
                    float d = 0.0f;
#pragma unroll
                    for (int m = 0; m < MK; ++m) d = fmaf(bf16_at(r_k, j * DK + lane + 32 * m), u[m], d);
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                    const float cf = r_be[j] * d, al = r_al[j];
#pragma unroll
                    for (int m = 0; m < MV; ++m) racc[m] = fmaf(cf, bf16_at(r_v, j * DV + lane + 32 * m), racc[m]);
#pragma unroll
                    for (int m = 0; m < MK; ++m) u[m] = al * fmaf(-cf, bf16_at(r_k, j * DK + lane + 32 * m), u[m]);
                }
#pragma unroll
                for (int m = 0; m < MK; ++m) s_u[ib * DK + lane + 32 * m] = u[m];
#pragma unroll
                for (int m = 0; m < MV; ++m) s_rt[ib * DV + lane + 32 * m] = racc[m];
            }
            if (work && ln + 1 >= L) gdn_fold_constants<DK>(s_fc + ib * kFcStride, r_k, r_al, ln + 1);
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull + ib);      // item kk is prepared
        }
        if (lane == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        return;
    }

    // ================================ consumer warps =================================
    const int ctid = tid - 64;                           // 0..255
    const int cw = ctid >> 5;                            // owns rows cw + RSTEP * v of each stage
    const int col4 = lane;                               // this lane's 4 columns
    bool live = true;
    int u = 0;                                           // stages consumed so far
    for (int w = 0; w < n_work; ++w) {
        const int k = s_list[w], r = w % RB, ib = w % kGdnBufs;
        if (live && !pwait(pfull + ib, (uint32_t)((w / kGdnBufs) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        if (live && !pwait(rfull + r, (uint32_t)((w / RB) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        const size_t bh = (size_t)item_of(k), cbh = cb_of(k);        // output, cache
        const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1];
        const bool work = live && !meta_bad(hd, ln);
        const bool fold = work && (ln + 1 >= L);
        const int nrec = ln + 1;
        const unsigned char *rb = rec(r);
        const uint16_t *r_k = reinterpret_cast<const uint16_t *>(rb + lay.rk_off);
        const uint16_t *r_v = reinterpret_cast<const uint16_t *>(rb + lay.rv_off);
        const float *r_al = reinterpret_cast<const float *>(rb + lay.ral_off);
        const float *r_be = reinterpret_cast<const float *>(rb + lay.rbe_off);
        const float4 u0 = *reinterpret_cast<const float4 *>(s_u + ib * DK + col4 * 4);
        const float *rt = s_rt + ib * DV;
        for (int uu = 0; uu < NU; ++uu, ++u) {
            const int s = u % S;
            if (live && !pwait(full + s, (uint32_t)((u / S) & 1), s_abort)) {
                live = false;
                *s_abort = 1;
            }
            const float4 *stg = reinterpret_cast<const float4 *>(stages + s * lay.stage_bytes);
            float4 hv[VPT];
#pragma unroll
            for (int v = 0; v < VPT; ++v) hv[v] = stg[ctid + v * NC];
            __syncwarp();                                // the warp is done with the stage
            if (lane == 0) mbar_arrive(empty + s);
            if (!work) continue;
            // o = S_c . u_0 + record term
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
                const int row = uu * kGdnRows + cw + RSTEP * reduced_index<G4, VPT>(0);
                a.o[bh * DV + row] = part[0] + rt[row];
            }
            if (fold)
                gdn_fold_stage<DK, DV, VPT>(hv, nrec, r_k, r_v, r_al, r_be, s_fc + ib * kFcStride,
                                            s_f + cw * (kGdnMaxRec * 8), uu, cw,
                                            reinterpret_cast<float4 *>(a.ckpt + (cbh * DV + uu * kGdnRows) * DK));
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(rempty + r);                     // record buffer r may be refilled
            mbar_arrive(pempty + ib);                    // and the item buffer ib
        }
    }
    if (ctid == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
}

}  // namespace rssm
