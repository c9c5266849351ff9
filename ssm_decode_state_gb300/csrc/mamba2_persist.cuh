// Persistent, warp-specialised, TMA-pipelined Mamba-2 replay decode (the
// serving-shape path: headdim 64, dstate 128, bf16 token inputs).
//
// One CTA per SM walks a static list of work items; an item is HPI heads of
// one group of one sequence.  At kernel start every thread block reads the
// ring pointers of all its items (and the last reader of a sequence commits
// the new ones); after that the warps never meet at a CTA-wide barrier:
//
//  * tile warp (warp 0, one lane): streams the checkpoint into an S-stage ring
//    of shared-memory buffers with one-dimensional bulk copies (the TMA
//    engine), completing on the stage's "full" mbarrier as transaction bytes:
//    one FP32 head tile (P x N) per stage, or on non-flush steps of a cache
//    with a read copy the FP8 codes and row scales of Q8 heads per stage (the
//    NVFP4 codes, block scales and row scales of Q4 heads).
//  * record warp (warp 1): copies each item's records (the used ring slots of
//    x and B are at most two contiguous runs each, plus the current token's x,
//    B and C, by bulk copy; dt words by cp.async) into a ring of RB record
//    buffers, RB items ahead of the consumers.
//  * preparation warps (warps 2 + NC/32 and up): per item, ahead of the
//    consumers, append the token to the ring, B_j . C_t, the decay weights and
//    the record term of every row, into triple-buffered item arrays handed
//    over through mbarriers.
//  * consumer warps (warps 2..): per stage, each warp reads its own 8 rows,
//    frees the stage, reduces the row dot products with C_t across its lanes
//    and writes y = exp(A S) (h_c . C_t) + record term; on flush steps it folds
//    h_c <- exp(A S) h_c + sum_j w_j x_j B_j^T into its rows and stores them
//    (and the FP8 copy).
//
// Every wait is bounded (~2 s, then RSSM_DEVERR_TIMEOUT and an orderly exit).
#pragma once

#include "mamba2_replay.cuh"
#include "persist_common.cuh"

namespace rssm {

struct PersistCfg {
    int items;     // B * H / HPI
    int max_my;    // items of the busiest CTA: ceil(items / grid)
    int nchunk;    // head chunks per group = hpg / HPI
    int stages;    // S: checkpoint tiles in flight
    int recbufs;   // RB: record buffers in flight
    int arrivals;  // items per sequence = H / HPI
    int stall;     // test hook: the consumers first wait on a barrier nothing arrives on
};

// Threads of a CTA: NC consumers + the tile warp and the record warp.
constexpr int persist_threads(int nc) { return nc + 64; }
// The decode kernel adds two item-preparation warps after the consumers.
constexpr int persist_decode_threads(int nc) { return nc + 64 + kPrepThreads; }

// Byte layout of the persistent kernel's shared memory.
// Heads whose FP8 codes share one stage (one wait, one release); the same
// count for NVFP4 copies (Q4).
__host__ __device__ constexpr int persist_q8(int hpi) { return hpi >= 4 ? 4 : hpi; }
__host__ __device__ constexpr int persist_q4(int hpi) { return hpi >= 4 ? 4 : hpi; }
// Heads per stage of an FP16 checkpoint read on non-flush steps.
__host__ __device__ constexpr int persist_q16(int hpi) { return hpi >= 2 ? 2 : 1; }

struct PSmem {
    int stage_bytes, stages_off;
    int full_off, empty_off, rfull_off, rempty_off;
    int rec_off, rx_off, rB_off, rC_off, rdt_off, rec_bytes;
    int meta_off, cb_off, w_off, decay_off, rt_off, wx_off, ad_off, flag_off, total;
    int pfull_off, pempty_off, wcb_off, sfx_off, cq_off, ch_off;
    // RC: read copy (0 none, 1 FP8, 2 NVFP4); CK: checkpoint precision (0 float32, 1 FP16)
    __host__ __device__ PSmem(int P, int N, int L, int HPI, int S, int RB, int H, int MY, int RC, int CK) {
        const int KM = L + 1;
        auto up = [](int v, int a) { return (v + a - 1) / a * a; };
        // one checkpoint tile (float32 or FP16), or the codes and row scales of
        // persist_q8(HPI) heads (FP8), or the codes, block scales and row scales of
        // persist_q4(HPI) heads (NVFP4)
        stage_bytes = CK ? persist_q16(HPI) * P * N * 2 : P * N * 4;
        if (RC == 1 && persist_q8(HPI) * (P * N + P * 4) > stage_bytes) stage_bytes = persist_q8(HPI) * (P * N + P * 4);
        if (RC == 2 && persist_q4(HPI) * (nv4_head_bytes(P, N) + P * 4) > stage_bytes)
            stage_bytes = persist_q4(HPI) * (nv4_head_bytes(P, N) + P * 4);
        int o = 0;
        stages_off = o; o += S * stage_bytes;
        full_off = o;   o += 8 * S;
        empty_off = o;  o += 8 * S;
        rfull_off = o;  o += 8 * RB;
        rempty_off = o; o += 8 * RB;
        pfull_off = o;  o += 8 * 3;
        pempty_off = o; o += 8 * 3;
        o = up(o, 128);
        // one record buffer: x [HPI][KM][P] bf16, B [KM][N] bf16, C [N] bf16, dt [HPI][KM] f32
        rx_off = 0;
        rB_off = up(HPI * KM * P * 2, 16);
        rC_off = rB_off + up(KM * N * 2, 16);
        rdt_off = rC_off + up(N * 2, 16);
        rec_bytes = up(rdt_off + HPI * KM * 4, 128);
        rec_off = o;   o += RB * rec_bytes;
        meta_off = o;  o += up(MY * 12, 16);                // [items of this CTA][head, len, cache slot]
        cb_off = o;    o += up(3 * KM * 4, 16);             // [3 items][KM]
        w_off = o;     o += up(3 * HPI * KM * 4, 16);       // [3][HPI][KM]
        decay_off = o; o += up(3 * HPI * 4, 16);            // [3][HPI]
        rt_off = o;    o += up(3 * HPI * P * 4, 16);        // [3][HPI][P] (rows owned per warp)
        wx_off = o;    o += up(KM * P * 4, 16);             // [KM][P]  (rows owned per warp)
        wcb_off = o;   o += up(3 * HPI * KM * 4, 16);       // [3][HPI][KM]  w_j (B_j . C_t)
        cq_off = o;    o += up(3 * N * 2, 16);              // [3][N] C_t (bf16) of the item
        ch_off = o;    o += up(3 * (N * 2 + 16), 16);       // [3] C_t for the read copies' products, then e
        sfx_off = o;   o += up(2 * HPI * (KM + 1) * 4, 16); // [2 warps][HPI][KM + 1] suffix sums (prep only)
        ad_off = o;    o += up(2 * H * 4, 16);              // A[H], D[H]
        flag_off = o;  o += 16;
        total = o;
    }
};

// RC: the cache's read copy (0 none, 1 FP8, 2 NVFP4), and CK: the checkpoint's
// precision (0 float32, 1 FP16 rounded stochastically at flushes), fixed per
// instantiation so that each holds only the paths it runs.
template <int N, int P, int VPT, int HPI, int RC, int CK>
__global__ void __launch_bounds__(persist_decode_threads(P * N / 4 / VPT), 1)
m2_decode_persistent(const M2Args a, const PersistCfg pc) {
    constexpr int kPConsumers = P * N / 4 / VPT;         // consumer threads
    constexpr int G4 = N / 4;                            // lanes per row
    constexpr int CX = P / 8, CB = N / 8;                // 16-byte chunks per x / B row
    constexpr int Q8 = persist_q8(HPI);                  // heads per stage of FP8 codes
    constexpr int Q4 = persist_q4(HPI);                  // heads per stage of NVFP4 codes
    constexpr int Q16 = persist_q16(HPI);                // heads per stage of FP16 tiles, non-flush steps
    constexpr int HB4 = nv4_head_bytes(P, N);            // one head's NVFP4 codes + block scales
    static_assert(G4 == 32 && VPT == 8 && kPConsumers / 32 * VPT == P, "a warp owns 8 whole consecutive rows");
    extern __shared__ __align__(128) unsigned char smraw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.L, H = a.H, G = a.G, hpg = a.hpg, KM = L + 1;
    const int S = pc.stages, RB = pc.recbufs;
    const PSmem lay(P, N, L, HPI, S, RB, H, pc.max_my, RC, CK);
    constexpr int TB = P * N * (CK ? 2 : 4);             // bytes of one checkpoint tile
    unsigned char *stages = smraw + lay.stages_off;
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + lay.full_off);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smraw + lay.empty_off);
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smraw + lay.rfull_off);
    uint64_t *rempty = reinterpret_cast<uint64_t *>(smraw + lay.rempty_off);
    int *s_meta = reinterpret_cast<int *>(smraw + lay.meta_off);
    float *s_cb = reinterpret_cast<float *>(smraw + lay.cb_off);
    float *s_w = reinterpret_cast<float *>(smraw + lay.w_off);
    float *s_decay = reinterpret_cast<float *>(smraw + lay.decay_off);
    float *s_rt = reinterpret_cast<float *>(smraw + lay.rt_off);
    float *s_wx = reinterpret_cast<float *>(smraw + lay.wx_off);
    float *s_A = reinterpret_cast<float *>(smraw + lay.ad_off), *s_D = s_A + H;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smraw + lay.flag_off);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smraw + lay.pfull_off);
    uint64_t *pempty = reinterpret_cast<uint64_t *>(smraw + lay.pempty_off);
    float *s_wcb = reinterpret_cast<float *>(smraw + lay.wcb_off);
    float *s_sfx = reinterpret_cast<float *>(smraw + lay.sfx_off);
    uint16_t *s_cq = reinterpret_cast<uint16_t *>(smraw + lay.cq_off);
    unsigned char *s_ch = smraw + lay.ch_off;

    const int grid = gridDim.x;
    const int n_my = (pc.items - (int)blockIdx.x + grid - 1) / grid;
    constexpr bool q8 = RC == 1, q4 = RC == 2;
    auto item_of = [&](int k) { return (int)blockIdx.x + k * grid; };
    auto item_b = [&](int it) { return it / (G * pc.nchunk); };      // item = (b * G + g) * nchunk + c
    auto item_h0 = [&](int it) {
        const int bg = it / pc.nchunk, c = it - bg * pc.nchunk;
        return (bg % G) * hpg + c * HPI;
    };
    auto meta_bad = [&](int hd, int ln) { return hd < 0 || hd >= L || ln < 0 || ln > L; };
    // a non-flush item of a cache with a read copy streams the FP8 codes, Q8 heads
    // per stage; every other item streams FP32 tiles, one head per stage
    auto fp8_item = [&](int hd, int ln) { return q8 && !meta_bad(hd, ln) && ln + 1 < L; };
    auto nv4_item = [&](int hd, int ln) { return q4 && !meta_bad(hd, ln) && ln + 1 < L; };
    // a non-flush item of an FP16 checkpoint without read copy: Q16 heads per stage
    auto h16_item = [&](int hd, int ln) { return CK && RC == 0 && !meta_bad(hd, ln) && ln + 1 < L; };
    // an item that folds: its consumers read its record buffer (x and B for the fold) and
    // release it; every other item's buffer is released by the preparation
    auto fold_item = [&](int hd, int ln) { return !meta_bad(hd, ln) && ln + 1 >= L; };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kPConsumers / 32);       // one arrival per consumer warp
        }
        for (int r = 0; r < RB; ++r) {
            mbar_init(rfull + r, 33);                    // 32 cp.async arrivals + lane 0's release
            mbar_init(rempty + r, kPConsumers / 32);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(pfull + i, 1);                     // the preparing warp's lane 0
            mbar_init(pempty + i, kPConsumers / 32);
        }
        *s_abort = 0;
        // the bounded-wait test's barrier (count 1, never arrived on), beside the flag
        if (pc.stall) mbar_init(reinterpret_cast<uint64_t *>(smraw + lay.flag_off + 8), 1);
        fence_mbar_init();
    }
    for (int i = tid; i < H; i += blockDim.x) {
        s_A[i] = a.A[i];
        s_D[i] = a.D[i];
    }
    // Ring pointers of every item of this CTA, read once here.  Each read is
    // followed by that item's arrival on its sequence's counter; the thread that
    // sees a sequence's last arrival commits the new pointers.  That is safe at
    // once: every item of the sequence, in every CTA, has read them already.
    for (int k = tid; k < n_my; k += blockDim.x) {
        const int it = item_of(k), b = item_b(it);
        const int sb = a.slots ? __ldg(a.slots + b) : b;     // the sequence's cache slot
        if (sb < 0 || sb >= a.cap) {                         // skipped by every warp role
            s_meta[k * 3 + 0] = -1;
            s_meta[k * 3 + 1] = 0;
            s_meta[k * 3 + 2] = 0;
            if (item_h0(it) == 0) flag_error(a.err, RSSM_DEVERR_SLOT);
            continue;
        }
        const int hd = __ldcg(a.ring_head + sb), ln = __ldcg(a.ring_len + sb);
        s_meta[k * 3 + 0] = hd;
        s_meta[k * 3 + 1] = ln;
        s_meta[k * 3 + 2] = sb;
        if (meta_bad(hd, ln) && item_h0(it) == 0) flag_error(a.err, RSSM_DEVERR_RING_META);
        __threadfence();
        if (atomicAdd(a.arrive + sb, 1) == pc.arrivals - 1) {
            __threadfence();
            if (!meta_bad(hd, ln)) {
                const bool fold = ln + 1 >= L;
                a.ring_head[sb] = fold ? (hd + ln + 1) % L : hd;
                a.ring_len[sb] = fold ? 0 : ln + 1;
            }
            a.arrive[sb] = 0;
        }
    }
    __syncthreads();                                     // the only CTA-wide barrier
    if (n_my <= 0) return;

    if (warp == 0) {
        // ================================= tile warp ==================================
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first_policy();
        bool ok = true;
        int issued = 0;                                  // stage units issued so far
        for (int k = 0; k < n_my && ok; ++k) {
            const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1];
            const bool f8 = fp8_item(hd, ln), f4 = nv4_item(hd, ln), f16 = h16_item(hd, ln);
            const int it = item_of(k), sb = s_meta[k * 3 + 2], h0 = item_h0(it);
            const int nu = f8 ? HPI / Q8 : f4 ? HPI / Q4 : f16 ? HPI / Q16 : HPI;
            for (int uu = 0; uu < nu; ++uu) {
                const int t = issued, s = t % S;
                if (t >= S) ok = pwait(empty + s, (uint32_t)(((t / S) - 1) & 1), s_abort) && !*s_abort;
                if (!ok) break;
                unsigned char *dst = stages + s * lay.stage_bytes;
                if (f4) {
                    // Q4 consecutive heads: their codes and block scales, then their row scales
                    const size_t hd0 = (size_t)sb * H + h0 + uu * Q4;
                    mbar_arrive_expect_tx(full + s, Q4 * (HB4 + P * 4));
                    bulk_g2s(dst, a.ckpt_q + hd0 * HB4, Q4 * HB4, full + s, pol);
                    bulk_g2s(dst + Q4 * HB4, a.ckpt_scale + hd0 * P, Q4 * P * 4, full + s, pol);
                } else if (f16) {
                    // Q16 consecutive heads' FP16 tiles, contiguous in the cache
                    const size_t tile = ((size_t)sb * H + h0 + uu * Q16) * P;
                    mbar_arrive_expect_tx(full + s, Q16 * TB);
                    bulk_g2s(dst, reinterpret_cast<const unsigned char *>(a.ckpt) + tile * N * 2, Q16 * TB, full + s, pol);
                } else if (!f8) {
                    const size_t tile = ((size_t)sb * H + h0 + uu) * P;
                    mbar_arrive_expect_tx(full + s, TB);
                    bulk_g2s(dst, reinterpret_cast<const unsigned char *>(a.ckpt) + tile * N * (CK ? 2 : 4), TB, full + s,
                             pol);
                } else {
                    // Q8 consecutive heads: their codes, then their row scales
                    const size_t tile = ((size_t)sb * H + h0 + uu * Q8) * P;
                    mbar_arrive_expect_tx(full + s, Q8 * (P * N + P * 4));
                    bulk_g2s(dst, a.ckpt_q + tile * N, Q8 * P * N, full + s, pol);
                    bulk_g2s(dst + Q8 * P * N, a.ckpt_scale + tile, Q8 * P * 4, full + s, pol);
                }
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
        const uint16_t *rx = static_cast<const uint16_t *>(a.rec_x);
        const uint16_t *rB = static_cast<const uint16_t *>(a.rec_B);
        const uint16_t *ix = static_cast<const uint16_t *>(a.x);
        const uint16_t *iB = static_cast<const uint16_t *>(a.Bin);
        const uint16_t *iC = static_cast<const uint16_t *>(a.Cin);
        bool ok = true;
        int k = 0;
        for (; k < n_my; ++k) {
            const int r = k % RB;
            if (lane == 0 && k >= RB) ok = pwait(rempty + r, (uint32_t)(((k / RB) - 1) & 1), s_abort) && !*s_abort;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const int it = item_of(k), b = item_b(it), h0 = item_h0(it), g = h0 / hpg;
            const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1], sb = s_meta[k * 3 + 2];
            const bool good = !meta_bad(hd, ln);
            if (good) {
                // records: list position j < ln is ring slot (hd + j) mod L, j = ln the current
                // token.  The used slots of a ring are at most two contiguous runs, copied
                // whole (x and B rows) by the TMA engine; dt words go by cp.async.
                unsigned char *rb = smraw + lay.rec_off + r * lay.rec_bytes;
                const int nrec = ln + 1;
                const int run1 = ln < L - hd ? ln : L - hd, run2 = ln - run1;
                if (lane == 0) mbar_arrive_expect_tx(rfull + r, (uint32_t)((HPI * nrec * P + nrec * N + N) * 2));
                __syncwarp();
                if (lane < HPI) {
                    const size_t bh = (size_t)sb * H + h0 + lane;      // cache
                    unsigned char *dx = rb + lay.rx_off + lane * KM * P * 2;
                    if (run1) bulk_g2s(dx, rx + (bh * L + hd) * P, run1 * P * 2, rfull + r);
                    if (run2) bulk_g2s(dx + run1 * P * 2, rx + bh * L * P, run2 * P * 2, rfull + r);
                    bulk_g2s(dx + ln * P * 2, ix + ((size_t)b * H + h0 + lane) * P, P * 2, rfull + r);
                } else if (lane == HPI) {
                    const size_t bg = (size_t)sb * G + g;              // cache
                    unsigned char *dB = rb + lay.rB_off;
                    if (run1) bulk_g2s(dB, rB + (bg * L + hd) * N, run1 * N * 2, rfull + r);
                    if (run2) bulk_g2s(dB + run1 * N * 2, rB + bg * L * N, run2 * N * 2, rfull + r);
                    bulk_g2s(dB + ln * N * 2, iB + ((size_t)b * G + g) * N, N * 2, rfull + r);
                } else if (lane == HPI + 1) {
                    bulk_g2s(rb + lay.rC_off, iC + ((size_t)b * G + g) * N, N * 2, rfull + r);
                }
                for (int idx = lane; idx < HPI * nrec; idx += 32) {
                    const int hh = idx / nrec, j = idx - hh * nrec;
                    const int slot = hd + j < L ? hd + j : hd + j - L;
                    cp_async4(rb + lay.rdt_off + (hh * KM + j) * 4,
                              j < ln ? a.rec_dt + ((size_t)sb * H + h0 + hh) * L + slot : a.dt + (size_t)b * H + h0 + hh);
                }
            }
            cp_async_arrive_noinc(rfull + r);
            if (lane == 0 && !good) mbar_arrive(rfull + r);   // with good metadata lane 0 arrived above
        }
        cp_async_wait_all();
        // the record copies of the last items may still be in flight: the CTA must
        // not end before they land (bounded waits; the consumers normally saw them)
        if (lane == 0)
            for (int kk = k - RB < 0 ? 0 : k - RB; kk < k; ++kk) mbar_wait(rfull + kk % RB, (uint32_t)((kk / RB) & 1));
        if (!ok && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        }
        return;
    }

    if (warp >= 2 + kPConsumers / 32) {
        // ============================ item-preparation warps ============================
        // Per item, ahead of the consumers: append the token to the ring, B_j . C_t,
        // the decay weights, and the record term of every row of every head.  The two
        // warps take alternate items (each item's chain of dependent steps is short of
        // work, so two items in flight double the rate).  Item arrays are
        // triple-buffered (ia = item % 3); pempty says the consumers are done with a
        // buffer, pfull hands a prepared one over.
        const int pw = (tid - 64 - kPConsumers) >> 5, ptid = lane;
        constexpr int PT = 32;                           // threads per item
        float *sfx = s_sfx + pw * HPI * (KM + 1);        // this warp's suffix sums
        bool live = true;
        for (int kk = pw; kk < n_my; kk += 2) {
            const int r = kk % RB, ia = kk % 3;
            // the preparation only writes the cache (the ring appends): b is the item's slot
            const int it = item_of(kk), b = s_meta[kk * 3 + 2], h0 = item_h0(it), g = h0 / hpg;
            if (live && kk >= 3 && !pwait(pempty + ia, (uint32_t)(((kk / 3) - 1) & 1), s_abort)) {
                live = false;
                *s_abort = 1;
            }
            if (live && !pwait(rfull + r, (uint32_t)((kk / RB) & 1), s_abort)) {
                live = false;
                *s_abort = 1;
            }
            const int hd = s_meta[kk * 3 + 0], ln = s_meta[kk * 3 + 1];
            const bool work = live && !meta_bad(hd, ln);
            const int nrec = ln + 1;
            const unsigned char *rb = smraw + lay.rec_off + r * lay.rec_bytes;
            const uint16_t *r_x = reinterpret_cast<const uint16_t *>(rb + lay.rx_off);
            const uint16_t *r_B = reinterpret_cast<const uint16_t *>(rb + lay.rB_off);
            const uint16_t *r_C = reinterpret_cast<const uint16_t *>(rb + lay.rC_off);
            const float *r_dt = reinterpret_cast<const float *>(rb + lay.rdt_off);
            float *cb = s_cb + ia * KM, *w = s_w + ia * HPI * KM, *wcb = s_wcb + ia * HPI * KM;
            float *dec = s_decay + ia * HPI, *rt = s_rt + ia * HPI * P;
            if (work && ln + 1 < L) {
                // a non-flush step appends the token to the ring, slot (hd + ln) mod L, which
                // no one reads during this launch; the token is already in the record buffer
                const int slot = hd + ln < L ? hd + ln : hd + ln - L;
                const int nBC = (h0 % hpg == 0) ? 2 * CB : 0;   // the group's first chunk writes B and C
                for (int idx = ptid; idx < HPI * CX + nBC + HPI; idx += PT) {
                    if (idx < HPI * CX) {
                        const int hh = idx / CX, c = idx - hh * CX;
                        const size_t bh = (size_t)b * H + h0 + hh;
                        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.rec_x) + (bh * L + slot) * P + c * 8) =
                            *reinterpret_cast<const uint4 *>(r_x + (hh * KM + ln) * P + c * 8);
                    } else if (idx < HPI * CX + nBC) {
                        const int rr = idx - HPI * CX;
                        const bool isC = rr >= CB;
                        const int c = isC ? rr - CB : rr;
                        uint16_t *dst = static_cast<uint16_t *>(isC ? a.rec_C : a.rec_B);
                        if (dst != nullptr)
                            *reinterpret_cast<uint4 *>(dst + ((((size_t)b * G + g) * L + slot) * N + c * 8)) =
                                *reinterpret_cast<const uint4 *>(isC ? r_C + c * 8 : r_B + ln * N + c * 8);
                    } else {
                        const int hh = idx - HPI * CX - nBC;
                        a.rec_dt[((size_t)b * H + h0 + hh) * L + slot] = r_dt[hh * KM + ln];
                    }
                }
            }
            if (work) {
                // suffix sums of dt per head, newest first (suffix_sum's order): one pass
                // per head gives every S_j and the total
                if (ptid < HPI) {
                    const float *dth = r_dt + ptid * KM;
                    float *sf = sfx + ptid * (KM + 1);
                    float acc = 0.0f;
                    for (int j = ln; j >= 0; --j) {
                        sf[j] = acc;
                        acc += dth[j];
                    }
                    sf[KM] = acc;
                }
                // B_j . C_t: 8 lanes per record, 16 columns per lane as bf16 pairs, then a
                // 3-level butterfly; 4 records at a time
                for (int jb = 0; jb < nrec; jb += 4) {
                    const int j = jb + (lane >> 3);
                    float acc = 0.0f;
                    if (j < nrec) {
                        const int c0 = (lane & 7) * 16;
                        const uint4 b0 = *reinterpret_cast<const uint4 *>(r_B + j * N + c0);
                        const uint4 b1 = *reinterpret_cast<const uint4 *>(r_B + j * N + c0 + 8);
                        const uint4 q0 = *reinterpret_cast<const uint4 *>(r_C + c0);
                        const uint4 q1 = *reinterpret_cast<const uint4 *>(r_C + c0 + 8);
                        acc = fma_bf16_pair(b0.x, q0.x, acc);
                        acc = fma_bf16_pair(b0.y, q0.y, acc);
                        acc = fma_bf16_pair(b0.z, q0.z, acc);
                        acc = fma_bf16_pair(b0.w, q0.w, acc);
                        acc = fma_bf16_pair(b1.x, q1.x, acc);
                        acc = fma_bf16_pair(b1.y, q1.y, acc);
                        acc = fma_bf16_pair(b1.z, q1.z, acc);
                        acc = fma_bf16_pair(b1.w, q1.w, acc);
                    }
                    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                    if (j < nrec && (lane & 7) == 0) cb[j] = acc;
                }
            }
            __syncwarp();                                // S_j and B_j . C_t
            if (work) {
                // w_j = exp(A S_j) dt_j, w_j (B_j . C_t), and exp(A S) per head
                for (int idx = ptid; idx < HPI * nrec; idx += PT) {
                    const int hh = idx / nrec, j = idx - hh * nrec;
                    const float wv = expf(s_A[h0 + hh] * sfx[hh * (KM + 1) + j]) * r_dt[hh * KM + j];
                    w[hh * KM + j] = wv;
                    wcb[hh * KM + j] = wv * cb[j];
                }
                if (ptid < HPI) dec[ptid] = expf(s_A[h0 + ptid] * sfx[ptid * (KM + 1) + KM]);
            }
            __syncwarp();                                // w, w (B . C)
            if (work) {
                // record term of every row: 8 consecutive rows of one head per thread
                for (int o = ptid; o < HPI * P / 8; o += PT) {
                    const int hh = o / (P / 8), r0 = (o - hh * (P / 8)) * 8;
                    const uint16_t *xh = r_x + hh * KM * P + r0;
                    const float *wc = wcb + hh * KM;
                    float acc[8];
#pragma unroll
                    for (int v = 0; v < 8; ++v) acc[v] = 0.0f;
                    for (int j = 0; j < nrec; ++j) {
                        const float c = wc[j];
                        const uint4 xr = *reinterpret_cast<const uint4 *>(xh + j * P);
                        acc[0] = fmaf(c, bf16lo(xr.x), acc[0]);
                        acc[1] = fmaf(c, bf16hi(xr.x), acc[1]);
                        acc[2] = fmaf(c, bf16lo(xr.y), acc[2]);
                        acc[3] = fmaf(c, bf16hi(xr.y), acc[3]);
                        acc[4] = fmaf(c, bf16lo(xr.z), acc[4]);
                        acc[5] = fmaf(c, bf16hi(xr.z), acc[5]);
                        acc[6] = fmaf(c, bf16lo(xr.w), acc[6]);
                        acc[7] = fmaf(c, bf16hi(xr.w), acc[7]);
                    }
                    const uint4 xl = *reinterpret_cast<const uint4 *>(xh + ln * P);
                    const float Dh = s_D[h0 + hh];
                    float4 *dst = reinterpret_cast<float4 *>(rt + hh * P + r0);
                    dst[0] = make_float4(fmaf(Dh, bf16lo(xl.x), acc[0]), fmaf(Dh, bf16hi(xl.x), acc[1]),
                                         fmaf(Dh, bf16lo(xl.y), acc[2]), fmaf(Dh, bf16hi(xl.y), acc[3]));
                    dst[1] = make_float4(fmaf(Dh, bf16lo(xl.z), acc[4]), fmaf(Dh, bf16hi(xl.z), acc[5]),
                                         fmaf(Dh, bf16lo(xl.w), acc[6]), fmaf(Dh, bf16hi(xl.w), acc[7]));
                }
            }
            // C_t goes with the item's arrays, so that the consumers of an item that does
            // not fold never read its record buffer: the preparation releases that buffer
            // itself and the record warp can run further ahead
            if (lane < N / 8)
                reinterpret_cast<uint4 *>(s_cq + ia * N)[lane] = reinterpret_cast<const uint4 *>(r_C)[lane];
            if constexpr (RC == 1) {
                // for the FP8 read path's E4M3 MMA: C_t 2^e as two E4M3 terms, hi = the
                // nearest E4M3 and lo = the nearest to 16 (C_t 2^e - hi), e set from the
                // item's largest |C_t| so that it lands in [2^7, 2^8) (E4M3 reaches 448).
                // A bf16 value within 2^-14 of that largest one is hi + lo / 16 exactly
                // (8 significant bits in two 4-bit terms); smaller ones keep an absolute
                // error below max|C_t| 2^-21.  Then e itself.
                static_assert(N == 128, "4 columns per lane");
                float cv[4], cmax = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cv[i] = bf16_at(r_C, lane * 4 + i);
                    cmax = fmaxf(cmax, fabsf(cv[i]));
                }
                cmax = group_max<32>(cmax);
                const int ce = cmax > 0.0f ? min(max(7 - ilogbf(cmax), -120), 120) : 0;
                const float cs = pow2f(ce);
#pragma unroll
                for (int i = 0; i < 4; ++i) cv[i] *= cs;
                const uint32_t hw = f32x4_to_e4m3x4(cv[0], cv[1], cv[2], cv[3]);
                uint32_t h01, h23;
                e4m3x4_to_f16x2(hw, h01, h23);
                const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
                const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
                const uint32_t lw = f32x4_to_e4m3x4((cv[0] - v01.x) * 16.0f, (cv[1] - v01.y) * 16.0f,
                                                    (cv[2] - v23.x) * 16.0f, (cv[3] - v23.y) * 16.0f);
                unsigned char *ch = s_ch + ia * (N * 2 + 16);
                reinterpret_cast<uint32_t *>(ch)[lane] = hw;
                reinterpret_cast<uint32_t *>(ch + N)[lane] = lw;
                if (lane == 0) *reinterpret_cast<int *>(ch + N * 2) = ce;
            } else if constexpr (RC == 2) {
                // for the NVFP4 read path: C_t as f16 pairs times 2^e, e set from the item's
                // largest |C_t| so that it lands just below 2^15 (exact and overflow-free;
                // only values below max|C_t| 2^-29 lose bits), and e itself
                static_assert(N == 128, "4 columns per lane");
                float cv[4], cmax = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cv[i] = bf16_at(r_C, lane * 4 + i);
                    cmax = fmaxf(cmax, fabsf(cv[i]));
                }
                cmax = group_max<32>(cmax);
                const int ce = cmax > 0.0f ? min(max(14 - ilogbf(cmax), -120), 120) : 0;
                const float cs = pow2f(ce);
                const __half2 p0 = __floats2half2_rn(cv[0] * cs, cv[1] * cs), p1 = __floats2half2_rn(cv[2] * cs, cv[3] * cs);
                unsigned char *ch = s_ch + ia * (N * 2 + 16);
                reinterpret_cast<uint2 *>(ch)[lane] =
                    make_uint2(*reinterpret_cast<const uint32_t *>(&p0), *reinterpret_cast<const uint32_t *>(&p1));
                if (lane == 0) *reinterpret_cast<int *>(ch + N * 2) = ce;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(pfull + ia);                 // item kk is prepared
                if (!fold_item(hd, ln)) mbar_arrive_n(rempty + r, kPConsumers / 32);
            }
        }
        if (ptid == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        return;
    }

    // ================================ consumer warps =================================
    const int ctid = tid - 64;                           // 0..255
    const int cw = ctid >> 5;                            // consumer warp: owns rows cw * VPT + v
    const int col4 = lane;                               // this lane's 4 columns
    bool live = true;                                    // false once any wait gave up

    int u = 0;                                           // stage units consumed so far
    for (int k = 0; k < n_my; ++k) {
        const int r = k % RB, ia = k % 3;
        const int it = item_of(k), b = item_b(it), h0 = item_h0(it), sb = s_meta[k * 3 + 2];
        const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1];
        // test hook of the failure path: a wait that runs out (nothing arrives on
        // this barrier), so that the abort below is taken on a healthy kernel
        if (k == 0 && pc.stall && live &&
            !pwait(reinterpret_cast<uint64_t *>(smraw + lay.flag_off + 8), 0u, s_abort)) {
            live = false;
            *s_abort = 1;
        }
        // the item's records and its prepared arrays
        if (live && !pwait(pfull + ia, (uint32_t)((k / 3) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        const bool fitem = fold_item(hd, ln);
        if (fitem && live && !pwait(rfull + r, (uint32_t)((k / RB) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        const bool work = live && !meta_bad(hd, ln);
        const bool fold = work && (ln + 1 >= L);
        const int nrec = ln + 1;
        const unsigned char *rb = smraw + lay.rec_off + r * lay.rec_bytes;
        const uint16_t *r_x = reinterpret_cast<const uint16_t *>(rb + lay.rx_off);
        const uint16_t *r_B = reinterpret_cast<const uint16_t *>(rb + lay.rB_off);
        const uint16_t *r_C = s_cq + ia * N;             // C_t, from the prepared item
        const float *w = s_w + ia * HPI * KM, *dec = s_decay + ia * HPI, *rt = s_rt + ia * HPI * P;
        const float4 cfr = make_float4(bf16_at(r_C, col4 * 4 + 0), bf16_at(r_C, col4 * 4 + 1),
                                       bf16_at(r_C, col4 * 4 + 2), bf16_at(r_C, col4 * 4 + 3));
        // y of head hh from its FP32 tile: h_c . C_t (rows reduced across the warp),
        // decayed, plus the record term
        auto head_y = [&](int hh, const float4 (&hv)[VPT]) {
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
                const int row = cw * VPT + reduced_index<G4, VPT>(0);
                a.y[((size_t)b * H + h0 + hh) * P + row] = fmaf(dec[hh], part[0], rt[hh * P + row]);
            }
        };
        if (h16_item(hd, ln)) {
            // FP16 checkpoint tiles of Q16 heads per stage: read this warp's rows of
            // every head, free the stage, then the heads' outputs
            for (int uu = 0; uu < HPI / Q16; ++uu, ++u) {
                const int s = u % S;
                if (live && !pwait(full + s, (uint32_t)((u / S) & 1), s_abort)) {
                    live = false;
                    *s_abort = 1;
                }
                const uint2 *stg = reinterpret_cast<const uint2 *>(stages + s * lay.stage_bytes);
                uint2 hw[Q16][VPT];
#pragma unroll
                for (int hq = 0; hq < Q16; ++hq) {
#pragma unroll
                    for (int v = 0; v < VPT; ++v) hw[hq][v] = stg[hq * (P * N / 4) + (cw * VPT + v) * G4 + lane];
                }
                __syncwarp();                            // the warp is done with the stage
                if (lane == 0) mbar_arrive(empty + s);
                if (!work) continue;
#pragma unroll
                for (int hq = 0; hq < Q16; ++hq) {
                    float4 hv[VPT];
#pragma unroll
                    for (int v = 0; v < VPT; ++v) hv[v] = f16x4_to_float4(hw[hq][v]);
                    head_y(uu * Q16 + hq, hv);
                }
            }
        } else if (nv4_item(hd, ln)) {
            // NVFP4 codes, Q4 heads per stage.  Lane (blk, rsub) takes the 16-column
            // block blk = lane & 7 of rows rsub and rsub + 4 (rsub = lane >> 3) of the
            // warp's 8 rows: its block sums need one block scale each, then the 8
            // lanes of a row reduce them.  Codes become f16 pairs in hardware; C_t
            // enters as f16 pairs times 2^e (prepared with the item), products are
            // exact, sums FP32 through the mixed-precision
            // fma.rn.f32.f16; 2^-e comes off at the end.  (Through the warp-level MMA,
            // with the block scales folded into A in f16, this step measured 85.9 us
            // against 82-83 us for this form: the per-k-tile byte extraction and
            // scale products cost more than the FMAs they replace.)
            const int blk = lane & 7, rsub = lane >> 3;
            // C_t as f16 x 2^e and e, prepared with the item: the block's column pairs
            const unsigned char *ch = s_ch + ia * (N * 2 + 16);
            const float cinv = pow2f(-*reinterpret_cast<const int *>(ch + N * 2));
            uint32_t cp[8];                              // pairs (2i, 2i + 1) of the block
            {
                const uint4 c0 = reinterpret_cast<const uint4 *>(ch)[2 * blk];
                const uint4 c1 = reinterpret_cast<const uint4 *>(ch)[2 * blk + 1];
                cp[0] = c0.x; cp[1] = c0.y; cp[2] = c0.z; cp[3] = c0.w;
                cp[4] = c1.x; cp[5] = c1.y; cp[6] = c1.z; cp[7] = c1.w;
            }
            for (int uu = 0; uu < HPI / Q4; ++uu, ++u) {
                const int s = u % S;
                if (live && !pwait(full + s, (uint32_t)((u / S) & 1), s_abort)) {
                    live = false;
                    *s_abort = 1;
                }
                const unsigned char *stg = stages + s * lay.stage_bytes;
                const float *sc = reinterpret_cast<const float *>(stg + Q4 * HB4);
                uint2 qc[Q4][2];
                uint32_t sbc[Q4][2];
#pragma unroll
                for (int hq = 0; hq < Q4; ++hq) {
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const int row = cw * VPT + rsub + 4 * m;
                        qc[hq][m] = *reinterpret_cast<const uint2 *>(stg + hq * HB4 + row * (N / 2) + blk * 8);
                        sbc[hq][m] = stg[hq * HB4 + P * N / 2 + row * (N / 16) + blk];
                    }
                }
                // the row scale of the (head, row) this lane ends up with after the reduction
                float rsv;
                {
                    const int vi = reduced_index<8, Q4 * 2>(0);
                    rsv = sc[(vi >> 1) * P + cw * VPT + rsub + 4 * (vi & 1)];
                }
                __syncwarp();                            // the warp is done with the stage
                if (lane == 0) mbar_arrive(empty + s);
                if (!work) continue;
                float part[Q4 * 2];
#pragma unroll
                for (int hq = 0; hq < Q4; ++hq) {
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        uint32_t pa[4], pb[4];
                        e2m1x8_to_f16x2(qc[hq][m].x, pa);
                        e2m1x8_to_f16x2(qc[hq][m].y, pb);
                        float acc = 0.0f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc = fma_f16_pair(pa[i], cp[i], acc);
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc = fma_f16_pair(pb[i], cp[4 + i], acc);
                        part[hq * 2 + m] = acc * e4m3_value(sbc[hq][m]);
                    }
                }
                group_reduce<8, Q4 * 2>(part);
                if (reduced_writer<8, Q4 * 2>()) {
                    const int vi = reduced_index<8, Q4 * 2>(0);
                    const int hh = uu * Q4 + (vi >> 1), row = cw * VPT + rsub + 4 * (vi & 1);
                    a.y[((size_t)b * H + h0 + hh) * P + row] =
                        fmaf(dec[hh], (part[0] * cinv) * rsv, rt[hh * P + row]);
                }
            }
        } else if (fp8_item(hd, ln)) {
            // FP8 codes, Q8 heads per stage: a warp's rows of the stage are its 8 rows of
            // each of the Q8 heads, and their products with C_t go through the warp-level
            // E4M3 MMA (m16n8k32, FP32 accumulation) as a matrix-vector product: the codes
            // are A as they are stored (rows x dstate, no conversion), and C_t 2^e, as two
            // E4M3 terms hi + lo / 16 (prepared with the item), is columns 0 (hi) and 1
            // (lo) of B, the other columns zero: one MMA forms both terms' sums, and
            // products are exact.  dstate is the MMA's reduction axis, so its order is
            // free: lane (g, t) = (lane >> 2, lane & 3) takes the 32 consecutive codes
            // 32 t .. 32 t + 31 of rows g and g + 8 of each 16-row tile, and k-tile kt
            // reads their bytes 8 kt .. 8 kt + 7 (a0 / a1 the first four, a2 / a3 the
            // next four); lanes 0-3 hold hi and lanes 4-7 lo in the same order.  2^-e
            // comes off at the end.  (Through the f16 MMA, each group of four codes first
            // took two conversions: the consumers' instructions bound the step; with a
            // separate MMA per term the tensor pipe took ~10 us of a 78 us step.)
            constexpr int MT = Q8 >= 2 ? Q8 / 2 : 1;       // 16-row tiles per warp and stage
            const int g = lane >> 2, t4 = lane & 3;
            const unsigned char *ch = s_ch + ia * (N * 2 + 16);
            const float cinv = pow2f(-*reinterpret_cast<const int *>(ch + N * 2));
            uint32_t bb[8];                              // B fragments: word 2 kt + (0, 1) of column g's term
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint4 w = g < 2 ? reinterpret_cast<const uint4 *>(ch + g * N)[t4 * 2 + q] : make_uint4(0u, 0u, 0u, 0u);
                bb[4 * q] = w.x; bb[4 * q + 1] = w.y; bb[4 * q + 2] = w.z; bb[4 * q + 3] = w.w;
            }
            for (int uu = 0; uu < HPI / Q8; ++uu, ++u) {
                const int s = u % S;
                if (live && !pwait(full + s, (uint32_t)((u / S) & 1), s_abort)) {
                    live = false;
                    *s_abort = 1;
                }
                const unsigned char *stg = stages + s * lay.stage_bytes;
                const float *sc = reinterpret_cast<const float *>(stg + Q8 * P * N);
                // rows g and g + 8 of tile mt are stage rows 16 mt + g (+ 8): head
                // (16 mt + g (+ 8)) / 8 of the stage, row cw * 8 + g of that head
                uint4 qv[MT][2][2];
                float rsv[MT][2];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                    for (int hv2 = 0; hv2 < 2; ++hv2) {
                        const int hq = 2 * mt + hv2;
                        if (hq < Q8) {
                            const unsigned char *rowp = stg + hq * (P * N) + (cw * VPT + g) * N + 32 * t4;
                            qv[mt][hv2][0] = *reinterpret_cast<const uint4 *>(rowp);
                            qv[mt][hv2][1] = *reinterpret_cast<const uint4 *>(rowp + 16);
                            rsv[mt][hv2] = sc[hq * P + cw * VPT + g];
                        } else {
                            qv[mt][hv2][0] = qv[mt][hv2][1] = make_uint4(0u, 0u, 0u, 0u);
                            rsv[mt][hv2] = 0.0f;
                        }
                    }
                }
                __syncwarp();                            // the warp is done with the stage
                if (lane == 0) mbar_arrive(empty + s);
                if (!work) continue;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint32_t w0[8] = {qv[mt][0][0].x, qv[mt][0][0].y, qv[mt][0][0].z, qv[mt][0][0].w,
                                            qv[mt][0][1].x, qv[mt][0][1].y, qv[mt][0][1].z, qv[mt][0][1].w};
                    const uint32_t w1[8] = {qv[mt][1][0].x, qv[mt][1][0].y, qv[mt][1][0].z, qv[mt][1][0].w,
                                            qv[mt][1][1].x, qv[mt][1][1].y, qv[mt][1][1].z, qv[mt][1][1].w};
                    // two accumulator sets (even and odd k-tiles): two short dependent chains
                    float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f, d3 = 0.0f, e0 = 0.0f, e1 = 0.0f, e2 = 0.0f, e3 = 0.0f;
#pragma unroll
                    for (int kt = 0; kt < 4; kt += 2) {
                        mma_e4m3_16x8x32(d0, d1, d2, d3, w0[2 * kt], w1[2 * kt], w0[2 * kt + 1], w1[2 * kt + 1],
                                         bb[2 * kt], bb[2 * kt + 1]);
                        mma_e4m3_16x8x32(e0, e1, e2, e3, w0[2 * kt + 2], w1[2 * kt + 2], w0[2 * kt + 3],
                                         w1[2 * kt + 3], bb[2 * kt + 2], bb[2 * kt + 3]);
                    }
                    // columns 0 (hi) and 1 (lo) of D: rows g (d0, d1) and g + 8 (d2, d3) in
                    // the lanes with t = 0
                    const float dh0 = d0 + e0, dl0 = d1 + e1, dh2 = d2 + e2, dl2 = d3 + e3;
                    if (t4 == 0) {
#pragma unroll
                        for (int hv2 = 0; hv2 < 2; ++hv2) {
                            const int hq = 2 * mt + hv2;
                            if (hq < Q8) {
                                const int hh = uu * Q8 + hq, row = cw * VPT + g;
                                const float dsum = hv2 ? fmaf(dl2, 0.0625f, dh2) : fmaf(dl0, 0.0625f, dh0);
                                a.y[((size_t)b * H + h0 + hh) * P + row] =
                                    fmaf(dec[hh], (dsum * cinv) * rsv[mt][hv2], rt[hh * P + row]);
                            }
                        }
                    }
                }
            }
        } else {
            for (int hh = 0; hh < HPI; ++hh, ++u) {
                const int s = u % S;
                if (live && !pwait(full + s, (uint32_t)((u / S) & 1), s_abort)) {
                    live = false;
                    *s_abort = 1;
                }
                float4 hv[VPT];
                if constexpr (CK) {
                    const uint2 *stg = reinterpret_cast<const uint2 *>(stages + s * lay.stage_bytes);
#pragma unroll
                    for (int v = 0; v < VPT; ++v) hv[v] = f16x4_to_float4(stg[(cw * VPT + v) * G4 + lane]);
                } else {
                    const float4 *stg = reinterpret_cast<const float4 *>(stages + s * lay.stage_bytes);
#pragma unroll
                    for (int v = 0; v < VPT; ++v) hv[v] = stg[(cw * VPT + v) * G4 + lane];
                }
                __syncwarp();                            // the warp is done with the stage
                if (lane == 0) mbar_arrive(empty + s);
                if (!work) continue;
                const size_t tile = ((size_t)sb * H + h0 + hh) * P;    // cache rows of this head
                if (fold) {
                    const float *wh = w + hh * KM;
                    const uint16_t *xh = r_x + hh * KM * P;
                    for (int idx = lane; idx < nrec * VPT; idx += 32) {
                        const int j = idx / VPT, v = idx - j * VPT, row = cw * VPT + v;
                        s_wx[j * P + row] = wh[j] * bf16_at(xh, j * P + row);
                    }
                    __syncwarp();
                }
                head_y(hh, hv);
                if (fold) {
                    // rank-nrec update first (each B_j loaded once per lane), then the
                    // decayed checkpoint in one fma: the state is rounded once per flush
                    unsigned long long acc01[VPT], acc23[VPT];      // packed (x, y) and (z, w)
#pragma unroll
                    for (int v = 0; v < VPT; ++v) acc01[v] = acc23[v] = 0ull;
                    for (int j = 0; j < nrec; ++j) {
                        const uint2 braw = *reinterpret_cast<const uint2 *>(r_B + j * N + col4 * 4);
                        const unsigned long long b01 = f2pack(bf16lo(braw.x), bf16hi(braw.x));
                        const unsigned long long b23 = f2pack(bf16lo(braw.y), bf16hi(braw.y));
                        // the warp's 8 consecutive rows: two 16-byte broadcast loads
                        const float4 wa = *reinterpret_cast<const float4 *>(s_wx + j * P + cw * VPT);
                        const float4 wb = *reinterpret_cast<const float4 *>(s_wx + j * P + cw * VPT + 4);
                        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                        for (int v = 0; v < VPT; ++v) {
                            const unsigned long long cc = f2pack(wv[v], wv[v]);
                            acc01[v] = fma2(cc, b01, acc01[v]);
                            acc23[v] = fma2(cc, b23, acc23[v]);
                        }
                    }
                    const float dk = dec[hh];
                    const unsigned long long dd = f2pack(dk, dk);
                    float4 o[VPT];
#pragma unroll
                    for (int v = 0; v < VPT; ++v) {
                        f2unpack(fma2(dd, f2pack(hv[v].x, hv[v].y), acc01[v]), o[v].x, o[v].y);
                        f2unpack(fma2(dd, f2pack(hv[v].z, hv[v].w), acc23[v]), o[v].z, o[v].w);
                    }
                    if constexpr (CK) {
                        // stochastic rounding to FP16; o[v] becomes the stored values.  One
                        // generator call serves the 8 columns of a lane pair: the even lane
                        // draws rows 2m, the odd lane rows 2m + 1, and each passes its
                        // partner the partner's two words of the row
                        const bool odd = lane & 1;
                        uint2 *ck2 = reinterpret_cast<uint2 *>(a.ckpt) + tile * N / 4;
#pragma unroll
                        for (int m = 0; m < VPT / 2; ++m) {
                            const uint4 r = philox4x32_10(
                                make_uint4((uint32_t)(lane >> 1), (uint32_t)(cw * VPT + 2 * m + odd),
                                           (uint32_t)(h0 + hh), (uint32_t)sb), a.seed_lo, a.seed_hi);
                            const uint32_t g0 = __shfl_xor_sync(0xffffffffu, odd ? r.x : r.z, 1);
                            const uint32_t g1 = __shfl_xor_sync(0xffffffffu, odd ? r.y : r.w, 1);
                            // select the words first: one rounding call per row for every lane
                            const int v0 = 2 * m, v1 = 2 * m + 1;
                            const uint32_t a0 = odd ? g0 : r.x, a1 = odd ? g1 : r.y;
                            const uint32_t b0 = odd ? r.z : g0, b1 = odd ? r.w : g1;
                            __stcs(ck2 + (cw * VPT + v0) * G4 + lane, sr_f16x4_words(o[v0], a0, a1));
                            __stcs(ck2 + (cw * VPT + v1) * G4 + lane, sr_f16x4_words(o[v1], b0, b1));
                        }
                    } else {
#pragma unroll
                        for (int v = 0; v < VPT; ++v)
                            st_stream(reinterpret_cast<float4 *>(a.ckpt + tile * N) + (cw * VPT + v) * G4 + lane, o[v]);
                    }
                    if (q4) {
                        nv4_quantize_store(o, a.ckpt_q + ((size_t)sb * H + h0 + hh) * HB4, a.ckpt_scale + tile, P, N,
                                           [&](int v) { return cw * VPT + v; });
                    } else if (q8) {
                        uint32_t q[VPT];
                        float rs;
                        e4m3_quantize_rows<VPT>(o, q, rs);
                        uint32_t *ckq = reinterpret_cast<uint32_t *>(a.ckpt_q + tile * N);
#pragma unroll
                        for (int v = 0; v < VPT; ++v) ckq[(cw * VPT + v) * G4 + lane] = q[v];
                        if (reduced_writer<32, VPT>()) a.ckpt_scale[tile + cw * VPT + reduced_index<32, VPT>(0)] = rs;
                    }
                    __syncwarp();                        // s_wx is rewritten for the next head
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (fitem) mbar_arrive(rempty + r);          // record buffer r may be refilled
            mbar_arrive(pempty + ia);                    // and the item arrays ia
        }
    }
    if (ctid == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
}

}  // namespace rssm
