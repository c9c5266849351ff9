// The fused flush of the gated-delta-rule replay decode on the fifth-generation
// tensor cores (serving head shape dk = dv = 128, bf16 token inputs).
//
// A decode step whose sequence has L - 1 buffered records folds them and its
// token into the checkpoint: the flush of the method (AT Pulse, What happened and
// Technical analysis, core idea; Gated DeltaNet is one of the layer types it
// ships kernels for, Capabilities and access).  The step kernel at
// the end of this file takes those (sequence, head) items in a first phase
// (gdn_fold_phase: their output o = S_c u_0 + record term and their folded
// checkpoint) and the others in a second one (gdn_decode_phase), over the same
// shared memory.
//
// The fold is the re-associated form that the decode phase also runs on the
// CUDA cores (gdn_fold_stage, for more than 512 items per CTA): with
// p_j = s_c . k_j for the nrec records (token last), d_j = a_j p_j +
// sum_{i<j} C_ij e_i, e_j = beta_j (v_j[r] - alpha_j d_j), f_j = e_j g_j, the
// new row is A s_c + sum_j f_j k_j, where C_ij = (k_i . k_j) prod_{i<m<j}
// alpha_m and a_j, g_j, A are prefix, suffix and total products of alpha.  Its
// contractions run on the tensor core: P = S_c K^T (128 x 128 by 128 x nrec),
// the keys' Gram matrix K K^T, and U = F K (128 x nrec by nrec x 128), each
// float32 factor written as three bf16 terms (t1 + t2 + t3 = x exactly), the
// keys being bf16 already, so every product is exact and the sums run in the
// float32 accumulator in tensor memory.  The query direction u_0 rides along as
// three more columns of P, so o needs no pass of its own.  U of F's first term
// and U of its two small terms accumulate apart and are added in float32 by
// the threads: added inside the accumulator, the small terms cost the folded
// state about two units in the last place (measured), which the following
// updates then amplify.
//
// In the fold phase each CTA takes the folding items of its static item list.
// Warps:
//  * compute warps 0-7: per item, read the state (64 KiB, staged by the load
//    warp) into registers and write its three bf16 terms (the MMA's A
//    operand), one 64-column K-block after the other so that the MMAs of the
//    first start while the second is written; after the projection MMA, warps
//    0-3 (one tensor-memory lane quarter each, one row per thread) run the
//    recurrence of their row, write o and F's three terms, while warp 4 turns
//    the Gram matrix into C (handed to warps 0-3 through a named barrier) and
//    warps 4-7 write the keys transposed (the update's B operand); after the
//    update MMA all eight move U through shared memory into the register
//    layout of the state and store A s_c + U.
//  * load warp 8: bulk copies (TMA engine) of each item's records and state.
//  * preparation warp 9, ahead of the compute warps: the backward chain (u_0,
//    record term), the projection operand (keys, u_0's three terms), the
//    products of alpha.
//  * MMA warp 10: allocates tensor memory; one lane issues the MMAs.
//
// Every wait is bounded (~2 s, then RSSM_DEVERR_TIMEOUT and an orderly exit:
// the copies and MMAs in flight complete before tensor memory is freed).
#pragma once

#include "gdn_persist.cuh"
#include "tc_common.cuh"

namespace rssm {

// Invalidates an mbarrier so that its memory may hold something else (or a
// new barrier) afterwards.
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

constexpr int kFtCompute = 256;                          // compute threads
constexpr int kFtThreads = kFtCompute + 96;              // + load, preparation and MMA warps
constexpr int kFtRB = 2, kFtPB = 2;                      // record and prepared-item buffers
// tensor-memory columns: P, the Gram matrix, U of F's first term, U of its other two
constexpr int kFtCols = 512, kFtPCol = 0, kFtGCol = 32, kFtU1Col = 256, kFtU23Col = 384;
constexpr int kFtURow = 24;                              // rows of the projection operand holding u_0's terms
constexpr int kFtMaxMy = 512;                            // items per CTA the fold phase takes
// fold constants of a prepared item (floats): [20][20] the products of alpha
// between two records, turned into C in place; per record {a_j, g_j, beta_j,
// alpha_j}; the total product A
constexpr int kFtRecC = kGdnMaxRec * kGdnMaxRec, kFtTot = kFtRecC + 4 * kGdnMaxRec, kFtFcStride = kFtTot + 4;

// Byte layout of the fold phase's shared memory (offsets from a 1024-byte
// aligned base).
struct FTSmem {
    int stage_off, planes_off, pop_off, kt_off, rec_off, rec_bytes, rk_off, rv_off, rq_off, ral_off, rbe_off;
    int u_off, rt_off, fc_off, bar_off, misc_off, total;
    __host__ __device__ FTSmem(int L) {
        const int DK = 128, DV = 128, KM = L + 1;
        auto up = [](int v, int a) { return (v + a - 1) / a * a; };
        int o = 0;
        stage_off = o;  o += DV * DK * 4;                 // the state, float32
        planes_off = o; o += 3 * 2 * 16384;               // S's three terms; later F's, then U
        pop_off = o;    o += kFtPB * 2 * 4096;            // projection operand per prepared item: 32 rows, 2 K-blocks
        kt_off = o;     o += 16384;                       // update operand: 128 rows, K 32 of 64
        rk_off = 0;
        rv_off = up(KM * DK * 2, 16);
        rq_off = rv_off + up(KM * DV * 2, 16);
        ral_off = rq_off + up(DK * 2, 16);
        rbe_off = ral_off + up(KM * 4, 16);
        rec_bytes = up(rbe_off + KM * 4, 128);
        rec_off = o;    o += kFtRB * rec_bytes;
        u_off = o;      o += kFtPB * DK * 4;
        rt_off = o;     o += kFtPB * DV * 4;
        fc_off = o;     o += kFtPB * kFtFcStride * 4;
        bar_off = o;    o += 20 * 8;
        misc_off = o;   o += 16;                          // tensor-memory base, abort flag
        total = o;
    }
};

// The fold phase of a step: the nf folding items of s_list (indices into this
// CTA's static item list; s_meta holds their ring pointers as read at kernel
// start).  sm is the 1024-byte aligned base of the dynamic shared memory.
// Every thread of the CTA calls it; warps from kFtThreads / 32 on only join
// its barriers.
template <int DK, int DV>
__device__ __forceinline__ void gdn_fold_phase(const GPArgs &a, unsigned char *sm, const int *s_meta,
                                               const int *s_list, int nf) {
    static_assert(DK == 128 && DV == 128, "serving head shape");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.L, H = a.H;
    const FTSmem lay(L);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + lay.bar_off);
    uint64_t *sfull = bars + 0, *sempty = bars + 1, *rfull = bars + 2, *rempty = bars + 4, *pfull = bars + 6,
             *pempty = bars + 8, *opsP0 = bars + 10, *opsP1 = bars + 11, *mmaG = bars + 12, *mmaP = bars + 13,
             *opsU = bars + 14, *mmaU = bars + 15, *tdone = bars + 16;
    constexpr int kFtBars = 17;
    uint32_t *s_taddr = reinterpret_cast<uint32_t *>(sm + lay.misc_off);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + lay.misc_off + 4);
    float *s_u = reinterpret_cast<float *>(sm + lay.u_off);
    float *s_rt = reinterpret_cast<float *>(sm + lay.rt_off);
    float *s_fc = reinterpret_cast<float *>(sm + lay.fc_off);
    unsigned char *planes = sm + lay.planes_off;
    auto rec = [&](int r) { return sm + lay.rec_off + r * lay.rec_bytes; };
    auto pop = [&](int pb) { return sm + lay.pop_off + pb * 8192; };

    const int grid = gridDim.x;
    auto item_of = [&](int k) { return (int)blockIdx.x + k * grid; };   // item = b * H + h

    if (tid == 0) {
        mbar_init(sfull, 1);
        mbar_init(sempty, 8);
        for (int r = 0; r < kFtRB; ++r) {
            mbar_init(rfull + r, 33);                    // 32 cp.async arrivals + lane 0's
            mbar_init(rempty + r, 8);
        }
        for (int i = 0; i < kFtPB; ++i) {
            mbar_init(pfull + i, 1);
            mbar_init(pempty + i, 8);
        }
        mbar_init(opsP0, 8);
        mbar_init(opsP1, 8);
        mbar_init(mmaG, 1);
        mbar_init(mmaP, 1);
        mbar_init(opsU, 8);
        mbar_init(mmaU, 1);
        mbar_init(tdone, 8);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 10) {
        tc::tmem_alloc(s_taddr, kFtCols);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t taddr = *s_taddr;
    auto cb_of = [&](int k) { return (size_t)s_meta[k * 3 + 2] * H + (size_t)(item_of(k) % H); };

    if (warp == 8) {
        // ================================= load warp ==================================
        const uint64_t pol = l2_evict_first_policy();
        bool ok = true;
        int nrecs = 0, nstates = 0;                      // items whose records / state were issued
        for (int i = 0; i < nf; ++i) {
            const int k = s_list[i], r = i % kFtRB;
            if (lane == 0 && i >= kFtRB) ok = pwait(rempty + r, (uint32_t)(((i / kFtRB) - 1) & 1), s_abort);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const size_t bh = (size_t)item_of(k), cbh = cb_of(k);
            const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1], nrec = ln + 1;
            const int run1 = ln < L - hd ? ln : L - hd, run2 = ln - run1;
            unsigned char *rb = rec(r);
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
            cp_async_arrive_noinc(rfull + r);
            nrecs = i + 1;
            // the state, once the compute warps hold the previous one in registers
            if (lane == 0 && i >= 1) ok = pwait(sempty, (uint32_t)((i - 1) & 1), s_abort);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(sfull, (uint32_t)(DV * DK * 4));
                bulk_g2s(sm + lay.stage_off, a.ckpt + cbh * DV * DK, DV * DK * 4, sfull, pol);
            }
            nstates = i + 1;
        }
        cp_async_wait_all();
        // copies of the last items may still be in flight: wait (bounded)
        if (lane == 0) {
            for (int kk = nrecs - kFtRB < 0 ? 0 : nrecs - kFtRB; kk < nrecs; ++kk)
                mbar_wait(rfull + kk % kFtRB, (uint32_t)((kk / kFtRB) & 1));
            if (nstates > 0) mbar_wait(sfull, (uint32_t)((nstates - 1) & 1));
        }
        if (!ok && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        }
    } else if (warp == 9) {
        // ============================== preparation warp ==============================
        bool live = true;
        for (int i = 0; i < nf; ++i) {
            const int k = s_list[i], r = i % kFtRB, pb = i % kFtPB;
            if (live && i >= kFtPB && !pwait(pempty + pb, (uint32_t)(((i / kFtPB) - 1) & 1), s_abort)) live = false;
            if (live && !pwait(rfull + r, (uint32_t)((i / kFtRB) & 1), s_abort)) live = false;
            if (!live) break;
            const int ln = s_meta[k * 3 + 1], nrec = ln + 1;
            const unsigned char *rb = rec(r);
            const uint16_t *r_k = reinterpret_cast<const uint16_t *>(rb + lay.rk_off);
            const uint16_t *r_v = reinterpret_cast<const uint16_t *>(rb + lay.rv_off);
            const uint16_t *r_q = reinterpret_cast<const uint16_t *>(rb + lay.rq_off);
            const float *r_al = reinterpret_cast<const float *>(rb + lay.ral_off);
            const float *r_be = reinterpret_cast<const float *>(rb + lay.rbe_off);
            // backward chain from the token: lane holds columns lane + 32 m of u and
            // rows lane + 32 m of the record term
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
            for (int m = 0; m < MK; ++m) s_u[pb * DK + lane + 32 * m] = u[m];
#pragma unroll
            for (int m = 0; m < MV; ++m) s_rt[pb * DV + lane + 32 * m] = racc[m];
            __syncwarp();
            // projection operand: rows j < nrec the keys, rows 24-26 u_0's three terms
            unsigned char *po = pop(pb);
            for (int idx = lane; idx < nrec * 16; idx += 32) {
                const int n = idx >> 4, c = idx & 15;
                *reinterpret_cast<uint4 *>(po + (c >> 3) * 4096 + tc::sw128_off(n, (c & 7) * 8)) =
                    *reinterpret_cast<const uint4 *>(r_k + n * DK + c * 8);
            }
            if (lane < 16) {
                const int c = lane;
                const float4 ua = *reinterpret_cast<const float4 *>(s_u + pb * DK + c * 8);
                const float4 ub = *reinterpret_cast<const float4 *>(s_u + pb * DK + c * 8 + 4);
                uint32_t t0[3], t1[3], t2[3], t3[3];
                tc::split3_bf16x2(ua.x, ua.y, t0[0], t0[1], t0[2]);
                tc::split3_bf16x2(ua.z, ua.w, t1[0], t1[1], t1[2]);
                tc::split3_bf16x2(ub.x, ub.y, t2[0], t2[1], t2[2]);
                tc::split3_bf16x2(ub.z, ub.w, t3[0], t3[1], t3[2]);
#pragma unroll
                for (int tt = 0; tt < 3; ++tt)
                    *reinterpret_cast<uint4 *>(po + (c >> 3) * 4096 + tc::sw128_off(kFtURow + tt, (c & 7) * 8)) =
                        make_uint4(t0[tt], t1[tt], t2[tt], t3[tt]);
            }
            // products of alpha: lane i's row of prod_{i<m<j} alpha_m, the prefix, suffix
            // and total products, each taken in increasing m
            float *fc = s_fc + pb * kFtFcStride;
            const float al = lane < nrec ? r_al[lane] : 1.0f, be = lane < nrec ? r_be[lane] : 0.0f;
            float pa = 1.0f, pre = 1.0f, suf = 1.0f, tot = 1.0f;
#pragma unroll
            for (int m = 0; m < kGdnMaxRec; ++m) {
                const float am = __shfl_sync(0xffffffffu, al, m);
                if (m < nrec) {
                    if (m > lane) {
                        fc[lane * kGdnMaxRec + m] = pa;
                        pa *= am;
                        suf *= am;
                    }
                    if (m < lane) pre *= am;
                    tot *= am;
                }
            }
            if (lane < nrec) *reinterpret_cast<float4 *>(fc + kFtRecC + 4 * lane) = make_float4(pre, suf, be, al);
            if (lane == 0) fc[kFtTot] = tot;
            tc::fence_async_smem();                      // the projection operand, for the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull + pb);
        }
        if (!live && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        }
    } else if (warp == 10) {
        // ================================= MMA warp ===================================
        uint64_t *last = nullptr;                        // the last commit's barrier and phase
        uint32_t last_par = 0;
        if (lane == 0) {
            const uint32_t pl = smem_u32(planes), kt = smem_u32(sm + lay.kt_off);
            auto give_up = [&]() {
                *s_abort = 1;
                flag_error(a.err, RSSM_DEVERR_TIMEOUT);
            };
            for (int i = 0; i < nf; ++i) {
                const int k = s_list[i], pb = i % kFtPB;
                const int nks = s_meta[k * 3 + 1] + 1 > 16 ? 2 : 1;
                const uint32_t po = smem_u32(pop(pb));
                const uint32_t par = (uint32_t)(i & 1);
                // the keys' Gram matrix, once the preparation warp wrote the operand: the
                // projection operand times itself (as A, the 128-row tile reads 96 rows
                // past the operand, inside this CTA's shared memory; their rows of the
                // product are never read)
                if (!pwait(pfull + pb, (uint32_t)((i / kFtPB) & 1), s_abort)) { give_up(); break; }
                tc::fence_after();
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint64_t kd = tc::sw128_desc(po + (kk >> 2) * 4096 + (kk & 3) * 32);
                    tc::mma_bf16(taddr + kFtGCol, kd, kd, tc::idesc_bf16(128, 32), kk > 0);
                }
                tc::mma_commit(mmaG);
                last = mmaG;
                last_par = par;
                // P = S_c K^T (and S_c u_0's terms), K-block by K-block as the terms land
                bool ok = true;
#pragma unroll 1
                for (int kb = 0; kb < 2 && ok; ++kb) {
                    if (!pwait(kb ? opsP1 : opsP0, par, s_abort)) { ok = false; break; }
                    tc::fence_after();
#pragma unroll 1
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_bf16(taddr + kFtPCol, tc::sw128_desc(pl + p * 32768 + kb * 16384 + ks * 32),
                                         tc::sw128_desc(po + kb * 4096 + ks * 32), tc::idesc_bf16(128, 32),
                                         kb > 0 || p > 0 || ks > 0);
                }
                if (!ok) { give_up(); break; }
                tc::mma_commit(mmaP);
                last = mmaP;
                if (!pwait(opsU, par, s_abort)) { give_up(); break; }
                tc::fence_after();
#pragma unroll 1
                for (int p = 0; p < 3; ++p)
                    for (int ks = 0; ks < nks; ++ks)
                        tc::mma_bf16(taddr + (p == 0 ? kFtU1Col : kFtU23Col), tc::sw128_desc(pl + p * 16384 + ks * 32),
                                     tc::sw128_desc(kt + ks * 32), tc::idesc_bf16(128, DK), p == 2 || ks > 0);
                tc::mma_commit(mmaU);
                last = mmaU;
            }
            // the MMAs in flight complete before tensor memory is freed
            if (last) mbar_wait(last, last_par);
            mbar_wait(tdone, 0);                         // and the compute warps' last loads
        }
        __syncwarp();
        tc::fence_after();
        tc::tmem_dealloc(taddr, kFtCols);
    } else if (warp < 8) {
        // ================================ compute warps ================================
        // thread (cw, lane) holds rows cw + 16 v + 8 (lane / 16) (v < 8), columns
        // 4 (lane % 16) .. + 3 of each 64-column K-block
        const int cw = warp, ctid = tid, half = lane >> 4, c16 = lane & 15;
        const int q4 = cw & 3;                           // tensor-memory lane quarter of this warp
        const float4 *stg = reinterpret_cast<const float4 *>(sm + lay.stage_off);
        float *scr = reinterpret_cast<float *>(planes);  // U in float32, [128][128], chunks swizzled by row
        bool live = true;
        auto cwait = [&](uint64_t *bar, uint32_t par) {
            if (live && !pwait(bar, par, s_abort)) {
                live = false;
                *s_abort = 1;
            }
        };
        for (int i = 0; i < nf; ++i) {
            const int k = s_list[i], r = i % kFtRB, pb = i % kFtPB;
            const int ln = s_meta[k * 3 + 1], nrec = ln + 1;
            const size_t bh = (size_t)item_of(k), cbh = cb_of(k);
            const uint32_t par = (uint32_t)(i & 1);
            cwait(sfull, par);
            float4 hv[16];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const int row = cw + 16 * v + 8 * half;
                hv[v] = stg[row * 32 + c16];
                hv[8 + v] = stg[row * 32 + 16 + c16];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sempty);          // the load warp may stage the next state
            // S's three bf16 terms, K-block 0 then K-block 1
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                if (live) {
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const float4 x = hv[8 * kb + v];
                        uint32_t a0, a1, a2, b0, b1, b2;
                        tc::split3_bf16x2(x.x, x.y, a0, a1, a2);
                        tc::split3_bf16x2(x.z, x.w, b0, b1, b2);
                        unsigned char *dst = planes + kb * 16384 + tc::sw128_off(cw + 16 * v + 8 * half, 4 * c16);
                        *reinterpret_cast<uint2 *>(dst) = make_uint2(a0, b0);
                        *reinterpret_cast<uint2 *>(dst + 32768) = make_uint2(a1, b1);
                        *reinterpret_cast<uint2 *>(dst + 65536) = make_uint2(a2, b2);
                    }
                    tc::fence_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(kb ? opsP1 : opsP0);
            }
            cwait(pfull + pb, (uint32_t)((i / kFtPB) & 1));
            cwait(rfull + r, (uint32_t)((i / kFtRB) & 1));
            const unsigned char *rb = rec(r);
            const uint16_t *r_k = reinterpret_cast<const uint16_t *>(rb + lay.rk_off);
            const uint16_t *r_v = reinterpret_cast<const uint16_t *>(rb + lay.rv_off);
            float *fc = s_fc + pb * kFtFcStride;
            const float A = fc[kFtTot];
            if (cw == 4) {
                // C_ij = (k_i . k_j) prod_{i<m<j} alpha_m from the Gram matrix (lane i holds row i)
                cwait(mmaG, par);
                tc::fence_after();
                if (live) {
                    float g[32];
                    tc::tmem_ld32(taddr + kFtGCol, g);
#pragma unroll
                    for (int j = 0; j < kGdnMaxRec; ++j)
                        if (j > lane && j < nrec) fc[lane * kGdnMaxRec + j] = g[j] * fc[lane * kGdnMaxRec + j];
                }
                tc::fence_before();
                asm volatile("bar.arrive 2, 160;" ::: "memory");   // to warps 0-3
            }
            if (live && cw >= 4) {
                // the update's B operand: keys transposed, row n = column n of the keys,
                // records 0 .. 31 (zero past nrec)
                const int n = ctid - 128, nch = nrec > 16 ? 4 : 2;
                for (int ch = 0; ch < nch; ++ch) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
                        const uint32_t lo = j0 < nrec ? r_k[j0 * DK + n] : 0u;
                        const uint32_t hi = j1 < nrec ? r_k[j1 * DK + n] : 0u;
                        w[e] = lo | (hi << 16);
                    }
                    *reinterpret_cast<uint4 *>(sm + lay.kt_off + tc::sw128_off(n, ch * 8)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                tc::fence_async_smem();
            }
            if (cw < 4) asm volatile("bar.sync 2, 160;" ::: "memory");   // C
            cwait(mmaP, par);
            tc::fence_after();
            if (live && cw < 4) {
                // one row per thread: P's row, o, the recurrence, F's three terms
                const int row = 32 * cw + lane;
                float p[32];
                tc::tmem_ld32(taddr + ((uint32_t)(32 * cw) << 16) + kFtPCol, p);
                a.o[bh * DV + row] = (p[kFtURow] + p[kFtURow + 1]) + p[kFtURow + 2] + s_rt[pb * DV + row];
                float acc[kGdnMaxRec], f[kGdnMaxRec];
#pragma unroll
                for (int m = 0; m < kGdnMaxRec; ++m) acc[m] = f[m] = 0.0f;
#pragma unroll
                for (int j = 0; j < kGdnMaxRec; ++j) {
                    if (j < nrec) {
                        const float4 cj = *reinterpret_cast<const float4 *>(fc + kFtRecC + 4 * j);   // a, g, beta, alpha
                        const float dj = fmaf(cj.x, p[j], acc[j]);
                        const float ej = cj.z * fmaf(-cj.w, dj, bf16_at(r_v, j * DV + row));
                        f[j] = ej * cj.y;
                        // row j of C, four at a time (rows are 16-byte aligned)
#pragma unroll
                        for (int m4 = (j + 1) / 4; m4 < kGdnMaxRec / 4; ++m4) {
                            const float4 cc = *reinterpret_cast<const float4 *>(fc + j * kGdnMaxRec + 4 * m4);
                            const float cv[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (4 * m4 + e > j) acc[4 * m4 + e] = fmaf(cv[e], ej, acc[4 * m4 + e]);
                        }
                    }
                }
                const int nch = nrec > 16 ? 4 : 2;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    if (ch >= nch) break;
                    uint32_t t[4][3];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;   // records past kGdnMaxRec are zero
                        tc::split3_bf16x2(j0 < kGdnMaxRec ? f[j0] : 0.0f, j1 < kGdnMaxRec ? f[j1] : 0.0f, t[e][0],
                                          t[e][1], t[e][2]);
                    }
#pragma unroll
                    for (int pp = 0; pp < 3; ++pp)
                        *reinterpret_cast<uint4 *>(planes + pp * 16384 + tc::sw128_off(row, ch * 8)) =
                            make_uint4(t[0][pp], t[1][pp], t[2][pp], t[3][pp]);
                }
                tc::fence_async_smem();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(opsU);
                mbar_arrive(rempty + r);                 // records and prepared item no longer read
                mbar_arrive(pempty + pb);
            }
            cwait(mmaU, par);
            tc::fence_after();
            if (live) {
                // U's rows 32 q4 + lane, columns 64 (cw / 4) .. + 63, into the scratch
                const int row = 32 * q4 + lane;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c0 = 64 * (cw >> 2) + 32 * h;
                    float uv[32], us[32];
                    tc::tmem_ld32(taddr + ((uint32_t)(32 * q4) << 16) + kFtU23Col + c0, us);
                    tc::tmem_ld32(taddr + ((uint32_t)(32 * q4) << 16) + kFtU1Col + c0, uv);
#pragma unroll
                    for (int j = 0; j < 32; ++j) uv[j] += us[j];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int ch = (c0 >> 2) + e;
                        *reinterpret_cast<float4 *>(scr + row * DK + ((ch ^ (row & 31)) << 2)) =
                            make_float4(uv[4 * e], uv[4 * e + 1], uv[4 * e + 2], uv[4 * e + 3]);
                    }
                }
            }
            tc::fence_before();
            consumer_sync<kFtCompute>();
            if (live) {
                // the folded rows: A s_c + U, in the layout the state was read in
                float4 *ck4 = reinterpret_cast<float4 *>(a.ckpt + cbh * DV * DK);
                const unsigned long long tt = f2pack(A, A);
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    const int row = cw + 16 * (v & 7) + 8 * half, ch = 16 * (v >> 3) + c16;
                    const float4 uu = *reinterpret_cast<const float4 *>(scr + row * DK + ((ch ^ (row & 31)) << 2));
                    float4 o;
                    f2unpack(fma2(tt, f2pack(hv[v].x, hv[v].y), f2pack(uu.x, uu.y)), o.x, o.y);
                    f2unpack(fma2(tt, f2pack(hv[v].z, hv[v].w), f2pack(uu.z, uu.w)), o.z, o.w);
                    st_stream(ck4 + row * 32 + ch, o);
                }
            }
            consumer_sync<kFtCompute>();                 // the scratch is free for the next item
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(tdone);
        if (ctid == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
    }
    // the phase is over (its copies and MMAs have completed): its barriers give
    // their memory back before the next phase lays out its own
    __syncthreads();
    if (tid == 0)
        for (int b = 0; b < kFtBars; ++b) mbar_inval(bars + b);
    __syncthreads();
}

// Shared memory of a step: the larger of the two phases' layouts, then the
// per-item ring pointers and the two item lists (1024 bytes of slack to align
// the base).
struct GStepSmem {
    int meta_off, flist_off, dlist_off, cnt_off, total;
    __host__ __device__ GStepSmem(int L, int S, int RB, int MY, bool fold_phase) {
        auto up = [](int v, int a) { return (v + a - 1) / a * a; };
        int core = GPSmem(128, 128, L, S, RB).total;
        if (fold_phase) {
            const int f = FTSmem(L).total;
            core = core > f ? core : f;
        }
        int o = up(core, 16);
        meta_off = o;  o += up(MY * 12, 16);               // [items of this CTA][head, len, cache slot]
        flist_off = o; o += up(MY * 4, 16);                // the folding items, in order
        dlist_off = o; o += up(MY * 4, 16);                // the others, in order
        cnt_off = o;   o += 16;
        total = o + 1024;
    }
};

// One decode step of the gated delta rule at the serving head shape (dk = dv =
// 128, bf16 token inputs), with the fused flush: one CTA per SM, a static list
// of (sequence, head) items per CTA.  The ring pointers of every item are read
// once at kernel start; the thread that sees a sequence's last arrival commits
// the new ones (every item of the sequence, in every CTA, has read them by
// then).  With a.skip_folds, the items whose sequence folds run first in the
// tensor-core fold phase, the rest in the decode phase; otherwise the decode
// phase takes every item and folds on the CUDA cores.
template <int DK, int DV>
__global__ void __launch_bounds__(256 + 64 + kPrepThreads, 1) gdn_decode_persistent(const GPArgs a) {
    extern __shared__ unsigned char gdraw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(gdraw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.L, H = a.H;
    const GStepSmem lay(L, a.stages, a.recbufs, a.max_my, a.skip_folds != 0);
    int *s_meta = reinterpret_cast<int *>(sm + lay.meta_off);
    int *s_flist = reinterpret_cast<int *>(sm + lay.flist_off);
    int *s_dlist = reinterpret_cast<int *>(sm + lay.dlist_off);
    int *s_cnt = reinterpret_cast<int *>(sm + lay.cnt_off);
    const int grid = gridDim.x;
    const int n_my = (a.items - (int)blockIdx.x + grid - 1) / grid;
    auto item_of = [&](int k) { return (int)blockIdx.x + k * grid; };   // item = b * H + h
    auto meta_bad = [&](int hd, int ln) { return hd < 0 || hd >= L || ln < 0 || ln > L; };

    for (int k = tid; k < n_my; k += blockDim.x) {
        const int it = item_of(k), b = it / H;
        const int sb = a.slots ? __ldg(a.slots + b) : b;     // the sequence's cache slot
        if (sb < 0 || sb >= a.cap) {                         // skipped by every warp role
            s_meta[k * 3 + 0] = -1;
            s_meta[k * 3 + 1] = 0;
            s_meta[k * 3 + 2] = 0;
            if (it % H == 0) flag_error(a.err, RSSM_DEVERR_SLOT);
            continue;
        }
        const int hd = __ldcg(a.ring_head + sb), ln = __ldcg(a.ring_len + sb);
        s_meta[k * 3 + 0] = hd;
        s_meta[k * 3 + 1] = ln;
        s_meta[k * 3 + 2] = sb;
        if (meta_bad(hd, ln) && it % H == 0) flag_error(a.err, RSSM_DEVERR_RING_META);
        __threadfence();
        if (atomicAdd(a.arrive + sb, 1) == H - 1) {
            __threadfence();
            if (!meta_bad(hd, ln)) {
                const bool fold = ln + 1 >= L;
                a.ring_head[sb] = fold ? (hd + ln + 1) % L : hd;
                a.ring_len[sb] = fold ? 0 : ln + 1;
            }
            a.arrive[sb] = 0;
        }
    }
    __syncthreads();
    // the two item lists (items with bad ring pointers go to the decode phase,
    // which skips them)
    if (warp == 0) {
        int nf = 0, nd = 0;
        for (int k0 = 0; k0 < n_my; k0 += 32) {
            const int k = k0 + lane;
            const int hd = k < n_my ? s_meta[k * 3 + 0] : 0, ln = k < n_my ? s_meta[k * 3 + 1] : 0;
            const bool f = k < n_my && a.skip_folds && !meta_bad(hd, ln) && ln + 1 >= L;
            const bool d = k < n_my && !f;
            const unsigned mf = __ballot_sync(0xffffffffu, f), md = __ballot_sync(0xffffffffu, d);
            const unsigned below = (1u << lane) - 1u;
            if (f) s_flist[nf + __popc(mf & below)] = k;
            if (d) s_dlist[nd + __popc(md & below)] = k;
            nf += __popc(mf);
            nd += __popc(md);
        }
        if (lane == 0) {
            s_cnt[0] = nf;
            s_cnt[1] = nd;
        }
    }
    __syncthreads();
    const int nf = s_cnt[0], nd = s_cnt[1];
    if (nf > 0) gdn_fold_phase<DK, DV>(a, sm, s_meta, s_flist, nf);
    if (nd > 0) gdn_decode_phase<DK, DV>(a, sm, s_meta, s_dlist, nd);
}

}  // namespace rssm
