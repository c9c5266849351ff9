// Persistent, warp-specialised speculative verify of T drafts (serving shapes).
//
// Same pipeline as the persistent decode (mamba2_persist.cuh): one CTA per SM,
// a tile warp streaming each head's FP32 checkpoint through shared-memory
// stages with bulk copies, a record warp copying each item's records (ring
// runs and the drafts, by bulk copy), two preparation warps and eight consumer
// warps that own whole rows.  Per item (HPI heads of one group of one
// sequence) the records are the len buffered ones plus the T drafts; draft i
// is scored against the checkpoint, the buffered records and drafts 1..i:
//   y_i = exp(A S_i) (h_c . C_i) + sum_{j <= len+i} exp(A (S_i - S_j)) dt_j (B_j . C_i) x_j + D x_i,
// with S the running sum of dt over the records.  If len + T > L the buffered
// records are first folded into the checkpoint (the pre-flush), with the same
// arithmetic as a flush; the outputs are read from the unfolded checkpoint
// plus all records, which is the same number.
//
// The preparation warps, ahead of the consumers, append the drafts' x and dt
// rows to the ring and compute B_j . C_i, the query weights and decays, the
// pre-flush fold weights and the record term of every (head, draft, row), into
// triple-buffered item arrays handed over through mbarriers.
//
// Ring pointers are read once at kernel start and committed there by the
// sequence's last arrival: pre-flush -> head <- (head + len) mod L, len <- T;
// otherwise len <- len + T.  The drafts' B and C rows are shared by the heads
// of a group and, on a pre-flush, land on slots other CTAs may still be
// reading, so a small epilogue kernel writes them after this one.
#pragma once

#include "mamba2_persist.cuh"

namespace rssm {

// Two-wide float32 product (sm_100+): each lane of the pair rounded once.
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Byte layout of the verify kernel's shared memory (T drafts, KM = L + T).
struct VSmem {
    int stage_bytes, stages_off;
    int full_off, empty_off, rfull_off, rempty_off, pfull_off, pempty_off;
    int rec_off, rx_off, rB_off, rC_off, rdt_off, rec_bytes;
    int meta_off, decay_off, wf_off, fdec_off, rt_off, cq_off, cb_off, wcb_off, sfx_off, sff_off, wx_off, ad_off, flag_off;
    int total;
    __host__ __device__ VSmem(int P, int N, int L, int T, int HPI, int S, int RB, int H, int MY) {
        const int KM = L + T;
        auto up = [](int v, int a) { return (v + a - 1) / a * a; };
        stage_bytes = P * N * 4;
        int o = 0;
        stages_off = o; o += S * stage_bytes;
        full_off = o;   o += 8 * S;
        empty_off = o;  o += 8 * S;
        rfull_off = o;  o += 8 * RB;
        rempty_off = o; o += 8 * RB;
        pfull_off = o;  o += 8 * 3;
        pempty_off = o; o += 8 * 3;
        o = up(o, 128);
        // one record buffer: x [HPI][KM][P] bf16, B [KM][N] bf16, C [T][N] bf16, dt [HPI][KM] f32
        rx_off = 0;
        rB_off = up(HPI * KM * P * 2, 16);
        rC_off = rB_off + up(KM * N * 2, 16);
        rdt_off = rC_off + up(T * N * 2, 16);
        rec_bytes = up(rdt_off + HPI * KM * 4, 128);
        rec_off = o;   o += RB * rec_bytes;
        meta_off = o;  o += up(MY * 12, 16);                // [items of this CTA][head, len, cache slot]
        // prepared items, triple-buffered
        decay_off = o; o += up(3 * HPI * T * 4, 16);        // [3][HPI][T]    exp(A S_i)
        wf_off = o;    o += up(3 * HPI * KM * 4, 16);       // [3][HPI][KM]   fold weights
        fdec_off = o;  o += up(3 * HPI * 4, 16);            // [3][HPI]       fold decay
        rt_off = o;    o += up(3 * HPI * T * P * 4, 16);    // [3][HPI][T][P] record terms
        cq_off = o;    o += up(3 * T * N * 2, 16);          // [3][T][N] the drafts' C (bf16)
        // the preparation warps' own scratch
        cb_off = o;    o += up(T * KM * 4, 16);             // [T][KM]        B_j . C_i
        wcb_off = o;   o += up(HPI * T * KM * 4, 16);       // [HPI][T][KM]   w_ij (B_j . C_i)
        sfx_off = o;   o += up(HPI * T * KM * 4, 16);       // [HPI][T][KM]   query suffix sums
        sff_off = o;   o += up(HPI * KM * 4, 16);           // [HPI][KM]      fold suffix sums
        wx_off = o;    o += up(KM * P * 4, 16);             // [KM][P] fold coefficients (rows owned per warp)
        ad_off = o;    o += up(2 * H * 4, 16);              // A[H], D[H]
        flag_off = o;  o += 16;
        total = o;
    }
};

template <int N, int P, int VPT, int HPI>
__global__ void __launch_bounds__(persist_decode_threads(P * N / 4 / VPT), 1)
m2_verify_persistent(const M2Args a, const PersistCfg pc) {
    constexpr int NC = P * N / 4 / VPT;                  // consumer threads
    constexpr int G4 = N / 4;                            // lanes per row
    constexpr int RSTEP = NC / G4;                       // rows between a thread's consecutive float4s
    constexpr int CX = P / 8;                            // 16-byte chunks per x row
    constexpr int TQ = 4;                                // draft slots in registers (T <= 4)
    static_assert(G4 == 32, "a warp owns whole rows");
    static_assert(HPI * TQ == 32 && TQ * VPT == 32, "one (head, draft) pair per lane");
    static_assert(HPI * TQ * 2 == kPrepThreads && HPI * (P / 8) == kPrepThreads,
                  "one (head, draft, half) and one (head, 8 rows) per preparation thread");
    extern __shared__ __align__(128) unsigned char smraw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.L, H = a.H, G = a.G, hpg = a.hpg, T = a.T, KM = L + T;
    const int S = pc.stages, RB = pc.recbufs;
    const VSmem lay(P, N, L, T, HPI, S, RB, H, pc.max_my);
    unsigned char *stages = smraw + lay.stages_off;
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + lay.full_off);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smraw + lay.empty_off);
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smraw + lay.rfull_off);
    uint64_t *rempty = reinterpret_cast<uint64_t *>(smraw + lay.rempty_off);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smraw + lay.pfull_off);
    uint64_t *pempty = reinterpret_cast<uint64_t *>(smraw + lay.pempty_off);
    int *s_meta = reinterpret_cast<int *>(smraw + lay.meta_off);
    float *s_cb = reinterpret_cast<float *>(smraw + lay.cb_off);
    float *s_wcb = reinterpret_cast<float *>(smraw + lay.wcb_off);
    float *s_sfx = reinterpret_cast<float *>(smraw + lay.sfx_off);
    float *s_sff = reinterpret_cast<float *>(smraw + lay.sff_off);
    float *s_decay = reinterpret_cast<float *>(smraw + lay.decay_off);
    float *s_wf = reinterpret_cast<float *>(smraw + lay.wf_off);
    float *s_fdec = reinterpret_cast<float *>(smraw + lay.fdec_off);
    float *s_rt = reinterpret_cast<float *>(smraw + lay.rt_off);
    float *s_wx = reinterpret_cast<float *>(smraw + lay.wx_off);
    uint16_t *s_cq = reinterpret_cast<uint16_t *>(smraw + lay.cq_off);
    float *s_A = reinterpret_cast<float *>(smraw + lay.ad_off), *s_D = s_A + H;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smraw + lay.flag_off);

    const int grid = gridDim.x;
    const int n_my = (pc.items - (int)blockIdx.x + grid - 1) / grid;
    auto item_of = [&](int k) { return (int)blockIdx.x + k * grid; };
    auto item_b = [&](int it) { return it / (G * pc.nchunk); };      // item = (b * G + g) * nchunk + c
    auto item_h0 = [&](int it) {
        const int bg = it / pc.nchunk, c = it - bg * pc.nchunk;
        return (bg % G) * hpg + c * HPI;
    };
    auto meta_bad = [&](int hd, int ln) { return hd < 0 || hd >= L || ln < 0 || ln > L; };
    // an item that pre-flushes: its consumers fold the buffered records (x and B from the
    // record buffer) and release that buffer; every other buffer the preparation releases
    auto pre_item = [&](int hd, int ln) { return !meta_bad(hd, ln) && ln + T > L; };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, NC / 32);       // one arrival per consumer warp
        }
        for (int r = 0; r < RB; ++r) {
            mbar_init(rfull + r, 33);                    // 32 cp.async arrivals + lane 0's release
            mbar_init(rempty + r, NC / 32);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(pfull + i, kPrepThreads / 32);     // one arrival per preparation warp
            mbar_init(pempty + i, NC / 32);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < H; i += blockDim.x) {
        s_A[i] = a.A[i];
        s_D[i] = a.D[i];
    }
    // ring pointers of every item, read once; the sequence's last arrival commits
    // the verify's pointers (pre-flush when the drafts would overflow the ring)
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
                const bool pre = ln + T > L;
                a.ring_head[sb] = pre ? (hd + ln) % L : hd;
                a.ring_len[sb] = (pre ? 0 : ln) + T;
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
        int issued = 0;
        for (int k = 0; k < n_my && ok; ++k) {
            const int it = item_of(k), sb = s_meta[k * 3 + 2], h0 = item_h0(it);
            for (int hh = 0; hh < HPI; ++hh) {
                const int t = k * HPI + hh, s = t % S;
                if (t >= S) ok = pwait(empty + s, (uint32_t)(((t / S) - 1) & 1), s_abort) && !*s_abort;
                if (!ok) break;
                const size_t tile = ((size_t)sb * H + h0 + hh) * P;
                mbar_arrive_expect_tx(full + s, P * N * 4);
                bulk_g2s(stages + s * lay.stage_bytes, a.ckpt + tile * N, P * N * 4, full + s, pol);
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
        // list position j < len: ring slot (hd + j) mod L; j = len + i: draft i
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
                // buffered records: at most two contiguous runs of ring slots; drafts: one
                // row each from the inputs; all by bulk copy, dt words by cp.async
                unsigned char *rb = smraw + lay.rec_off + r * lay.rec_bytes;
                const int nrec = ln + T;
                const int run1 = ln < L - hd ? ln : L - hd, run2 = ln - run1;
                if (lane == 0)
                    mbar_arrive_expect_tx(rfull + r, (uint32_t)((HPI * nrec * P + nrec * N + T * N) * 2));
                __syncwarp();
                if (lane < HPI) {
                    const size_t bh = (size_t)sb * H + h0 + lane;      // cache
                    unsigned char *dx = rb + lay.rx_off + lane * KM * P * 2;
                    if (run1) bulk_g2s(dx, rx + (bh * L + hd) * P, run1 * P * 2, rfull + r);
                    if (run2) bulk_g2s(dx + run1 * P * 2, rx + bh * L * P, run2 * P * 2, rfull + r);
                    for (int i = 0; i < T; ++i)
                        bulk_g2s(dx + (ln + i) * P * 2, ix + (((size_t)b * T + i) * H + h0 + lane) * P, P * 2, rfull + r);
                } else if (lane == HPI) {
                    const size_t bg = (size_t)sb * G + g;              // cache
                    unsigned char *dB = rb + lay.rB_off;
                    if (run1) bulk_g2s(dB, rB + (bg * L + hd) * N, run1 * N * 2, rfull + r);
                    if (run2) bulk_g2s(dB + run1 * N * 2, rB + bg * L * N, run2 * N * 2, rfull + r);
                    for (int i = 0; i < T; ++i)
                        bulk_g2s(dB + (ln + i) * N * 2, iB + (((size_t)b * T + i) * G + g) * N, N * 2, rfull + r);
                } else if (lane == HPI + 1) {
                    for (int i = 0; i < T; ++i)
                        bulk_g2s(rb + lay.rC_off + i * N * 2, iC + (((size_t)b * T + i) * G + g) * N, N * 2, rfull + r);
                }
                for (int idx = lane; idx < HPI * nrec; idx += 32) {
                    const int hh = idx / nrec, j = idx - hh * nrec;
                    const size_t bh = (size_t)sb * H + h0 + hh;        // cache
                    const int slot = hd + j < L ? hd + j : hd + j - L;
                    cp_async4(rb + lay.rdt_off + (hh * KM + j) * 4,
                              j < ln ? a.rec_dt + bh * L + slot : a.dt + ((size_t)b * T + (j - ln)) * H + h0 + hh);
                }
            }
            cp_async_arrive_noinc(rfull + r);
            if (lane == 0 && !good) mbar_arrive(rfull + r);   // with good metadata lane 0 arrived above
        }
        cp_async_wait_all();
        // the record copies of the last items may still be in flight: wait (bounded)
        if (lane == 0)
            for (int kk = k - RB < 0 ? 0 : k - RB; kk < k; ++kk) mbar_wait(rfull + kk % RB, (uint32_t)((kk / RB) & 1));
        if (!ok && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        }
        return;
    }

    if (warp >= 2 + NC / 32) {
        // ============================ item-preparation warps ============================
        const int ptid = tid - 64 - NC, pw = ptid >> 5;
        bool live = true;
        for (int kk = 0; kk < n_my; ++kk) {
            const int r = kk % RB, ia = kk % 3;
            // the preparation only writes the cache (the draft appends): b is the item's slot
            const int it = item_of(kk), b = s_meta[kk * 3 + 2], h0 = item_h0(it);
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
            const bool pre = ln + T > L;
            const unsigned char *rb = smraw + lay.rec_off + r * lay.rec_bytes;
            const uint16_t *r_x = reinterpret_cast<const uint16_t *>(rb + lay.rx_off);
            const uint16_t *r_B = reinterpret_cast<const uint16_t *>(rb + lay.rB_off);
            const uint16_t *r_C = reinterpret_cast<const uint16_t *>(rb + lay.rC_off);
            const float *r_dt = reinterpret_cast<const float *>(rb + lay.rdt_off);
            float *dec = s_decay + ia * HPI * T, *rt = s_rt + ia * HPI * T * P;
            float *wf = s_wf + ia * HPI * KM, *fdec = s_fdec + ia * HPI;
            if (work) {
                // drafts' x and dt rows into the ring (per head, read by no other CTA): thread
                // (head, draft, half) = (ptid / 8, ptid / 2 % 4, ptid % 2) copies half of the
                // draft's x row, thread (head, draft) = (ptid / 4, ptid % 4) its dt word
                const int hd2 = pre ? (hd + ln) % L : hd, ln2 = pre ? 0 : ln;
                {
                    const int hh = ptid >> 3, i = (ptid >> 1) & 3, half = ptid & 1;
                    if (i < T) {
                        const size_t bh = (size_t)b * H + h0 + hh;
                        const int slot = (hd2 + ln2 + i) % L;
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.rec_x) + (bh * L + slot) * P) +
                                     half * (CX / 2);
                        const uint4 *src = reinterpret_cast<const uint4 *>(r_x + (hh * KM + ln + i) * P) + half * (CX / 2);
#pragma unroll
                        for (int c = 0; c < CX / 2; ++c) dst[c] = src[c];
                    }
                    const int hd_ = ptid >> 2, id_ = ptid & 3;
                    if (ptid < HPI * TQ && id_ < T)
                        a.rec_dt[((size_t)b * H + h0 + hd_) * L + (hd2 + ln2 + id_) % L] = r_dt[hd_ * KM + ln + id_];
                }
                // suffix sums of dt, newest first (suffix_sum's order): one pass per
                // (head, draft) up to len + i gives that draft's S_ij and its decay;
                // one pass per head over the buffered records gives the fold's
                if (ptid < HPI * T) {
                    const int hh = ptid / T, i = ptid - hh * T;
                    const float *dth = r_dt + hh * KM;
                    float *sf = s_sfx + (hh * T + i) * KM;
                    float acc = 0.0f;
                    for (int j = ln + i; j >= 0; --j) {
                        sf[j] = acc;
                        acc += dth[j];
                    }
                    dec[hh * T + i] = expf(s_A[h0 + hh] * acc);
                } else if (pre && ptid < HPI * T + HPI) {
                    const int hh = ptid - HPI * T;
                    const float *dth = r_dt + hh * KM;
                    float *sf = s_sff + hh * KM;
                    float acc = 0.0f;
                    for (int j = ln - 1; j >= 0; --j) {
                        sf[j] = acc;
                        acc += dth[j];
                    }
                    fdec[hh] = expf(s_A[h0 + hh] * acc);
                }
                // B_j . C_i for every draft i and record j <= len + i (the valid pairs only,
                // draft-major): 8 lanes per pair, 16 columns per lane as bf16 pairs, then a
                // 3-level butterfly; each warp takes 4 pairs at a time
                const int npairs = T * (ln + 1) + T * (T - 1) / 2;
                for (int pb0 = pw * 4; pb0 < npairs; pb0 += 8) {
                    const int pr = pb0 + (lane >> 3);
                    const bool valid = pr < npairs;
                    int i = 0, j = pr;
                    while (valid && j >= ln + 1 + i) {
                        j -= ln + 1 + i;
                        ++i;
                    }
                    float acc = 0.0f;
                    if (valid) {
                        const int c0 = (lane & 7) * 16;
                        const uint4 b0 = *reinterpret_cast<const uint4 *>(r_B + j * N + c0);
                        const uint4 b1 = *reinterpret_cast<const uint4 *>(r_B + j * N + c0 + 8);
                        const uint4 q0 = *reinterpret_cast<const uint4 *>(r_C + i * N + c0);
                        const uint4 q1 = *reinterpret_cast<const uint4 *>(r_C + i * N + c0 + 8);
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
                    if (valid && (lane & 7) == 0) s_cb[i * KM + j] = acc;
                }
            }
            prep_sync();                                 // suffix sums and B . C
            if (work) {
                // query weights times B_j . C_i (valid pairs only: thread (head, draft, half)
                // takes records j = half, half + 2, .. <= len + i), and the pre-flush fold
                // weights (thread (head, part) records j = part, part + 8, .. < len)
                {
                    const int hh = ptid >> 3, i = (ptid >> 1) & 3, half = ptid & 1;
                    if (i < T) {
                        const float Ah = s_A[h0 + hh];
                        const float *sf = s_sfx + (hh * T + i) * KM;
                        float *wc = s_wcb + (hh * T + i) * KM;
                        for (int j = half; j <= ln + i; j += 2) {
                            const float wv = expf(Ah * sf[j]) * r_dt[hh * KM + j];
                            wc[j] = wv * s_cb[i * KM + j];
                        }
                    }
                    if (pre) {
                        const int part = ptid & 7;
                        for (int j = part; j < ln; j += 8)
                            wf[hh * KM + j] = expf(s_A[h0 + hh] * s_sff[hh * KM + j]) * r_dt[hh * KM + j];
                    }
                }
            }
            prep_sync();                                 // w (B . C)
            if (work) {
                // record terms: 8 consecutive rows of one head per thread, for every draft
                // (each x row loaded and converted once for the T drafts)
                const int hh = ptid >> 3, r0 = (ptid & 7) * 8;
                const uint16_t *xh = r_x + hh * KM * P + r0;
                const float *wch = s_wcb + hh * T * KM;
                float acc[TQ][8];
#pragma unroll
                for (int i = 0; i < TQ; ++i) {
#pragma unroll
                    for (int v = 0; v < 8; ++v) acc[i][v] = 0.0f;
                }
                for (int j = 0; j < ln + T; ++j) {
                    const uint4 xr = *reinterpret_cast<const uint4 *>(xh + j * P);
                    const float xv[8] = {bf16lo(xr.x), bf16hi(xr.x), bf16lo(xr.y), bf16hi(xr.y),
                                         bf16lo(xr.z), bf16hi(xr.z), bf16lo(xr.w), bf16hi(xr.w)};
#pragma unroll
                    for (int i = 0; i < TQ; ++i) {
                        if (i < T && j <= ln + i) {
                            const float c = wch[i * KM + j];
#pragma unroll
                            for (int v = 0; v < 8; ++v) acc[i][v] = fmaf(c, xv[v], acc[i][v]);
                        }
                    }
                }
                const float dh = s_D[h0 + hh];
#pragma unroll
                for (int i = 0; i < TQ; ++i) {
                    if (i < T) {
                        const uint4 xl = *reinterpret_cast<const uint4 *>(xh + (ln + i) * P);
                        float4 *dst = reinterpret_cast<float4 *>(rt + (hh * T + i) * P + r0);
                        dst[0] = make_float4(fmaf(dh, bf16lo(xl.x), acc[i][0]), fmaf(dh, bf16hi(xl.x), acc[i][1]),
                                             fmaf(dh, bf16lo(xl.y), acc[i][2]), fmaf(dh, bf16hi(xl.y), acc[i][3]));
                        dst[1] = make_float4(fmaf(dh, bf16lo(xl.z), acc[i][4]), fmaf(dh, bf16hi(xl.z), acc[i][5]),
                                             fmaf(dh, bf16lo(xl.w), acc[i][6]), fmaf(dh, bf16hi(xl.w), acc[i][7]));
                    }
                }
            }
            __syncwarp();
            // the drafts' C goes with the item's arrays, so that the consumers of an item
            // without a pre-flush never read its record buffer
            for (int c = ptid; c < T * N / 8; c += kPrepThreads)
                reinterpret_cast<uint4 *>(s_cq + ia * T * N)[c] = reinterpret_cast<const uint4 *>(r_C)[c];
            prep_sync();                                 // both warps are done with the buffer
            if (lane == 0) mbar_arrive(pfull + ia);      // item kk is prepared (one arrival per warp)
            if (ptid == 0 && !pre_item(hd, ln)) mbar_arrive_n(rempty + r, NC / 32);
        }
        if (ptid == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        return;
    }

    // ================================ consumer warps =================================
    const int ctid = tid - 64;                           // 0..NC-1
    const int cw = ctid >> 5;                            // consumer warp: owns rows cw + RSTEP * v
    const int col4 = lane;                               // this lane's 4 columns
    bool live = true;

    for (int k = 0; k < n_my; ++k) {
        const int r = k % RB, ia = k % 3;
        const int it = item_of(k), b = item_b(it), h0 = item_h0(it), sb = s_meta[k * 3 + 2];
        if (live && !pwait(pfull + ia, (uint32_t)((k / 3) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1];
        const bool pitem = pre_item(hd, ln);
        if (pitem && live && !pwait(rfull + r, (uint32_t)((k / RB) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        const bool work = live && !meta_bad(hd, ln);
        const bool pre = work && (ln + T > L);
        const unsigned char *rb = smraw + lay.rec_off + r * lay.rec_bytes;
        const uint16_t *r_x = reinterpret_cast<const uint16_t *>(rb + lay.rx_off);
        const uint16_t *r_B = reinterpret_cast<const uint16_t *>(rb + lay.rB_off);
        const uint16_t *r_C = s_cq + ia * T * N;         // the drafts' C, from the prepared item
        const float *dec = s_decay + ia * HPI * T, *rt = s_rt + ia * HPI * T * P;
        const float *wf = s_wf + ia * HPI * KM, *fdec = s_fdec + ia * HPI;
        // the drafts' C at this lane's 4 columns, as packed pairs (columns 0-1, 2-3).
        // Draft slot i holds draft i ^ ((lane / 8) % 4): the first two rounds of the
        // reduction below then trade the same half of every lane's values (no selects)
        unsigned long long cxy[TQ], czw[TQ];
#pragma unroll
        for (int i = 0; i < TQ; ++i) {
            const int di = i ^ ((lane >> 3) & 3);
            const bool on = di < T;
            cxy[i] = f2pack(on ? bf16_at(r_C, di * N + col4 * 4 + 0) : 0.f, on ? bf16_at(r_C, di * N + col4 * 4 + 1) : 0.f);
            czw[i] = f2pack(on ? bf16_at(r_C, di * N + col4 * 4 + 2) : 0.f, on ? bf16_at(r_C, di * N + col4 * 4 + 3) : 0.f);
        }
        for (int hh = 0; hh < HPI; ++hh) {
            const int t = k * HPI + hh, s = t % S;
            if (live && !pwait(full + s, (uint32_t)((t / S) & 1), s_abort)) {
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
            const int h = h0 + hh;
            const size_t tile = ((size_t)sb * H + h) * P;              // cache rows of this head
            // T x 8 row dot products reduced across the warp: lane ends with (draft, row)
            float part[TQ * VPT];
#pragma unroll
            for (int i = 0; i < TQ; ++i) {
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    // columns 0 + 2 and 1 + 3 as the two lanes of one packed pair
                    float lo, hi;
                    f2unpack(fma2(f2pack(hv[v].z, hv[v].w), czw[i], mul2(f2pack(hv[v].x, hv[v].y), cxy[i])), lo, hi);
                    part[i * VPT + v] = lo + hi;
                }
            }
            // reduce the 32 (draft slot, row) values across the warp: with the draft
            // slots permuted by lane bits 3-4, the rounds over lane bits 4 and 3 keep the
            // low half and trade the high half on every lane; then the usual exchange
            // over bits 2-0.  Lane l ends with draft l / 8, row l % 8 (as group_reduce)
            static_assert(G4 == 32 && TQ * VPT == 32, "one value per lane after the reduction");
#pragma unroll
            for (int q = 0; q < 16; ++q) part[q] += __shfl_xor_sync(0xffffffffu, part[q + 16], 16);
#pragma unroll
            for (int q = 0; q < 8; ++q) part[q] += __shfl_xor_sync(0xffffffffu, part[q + 8], 8);
            GroupReduce<4, 8, TQ * VPT>::run(part, lane);
            {
                const int vi = reduced_index<G4, TQ * VPT>(0);
                const int i = vi / VPT, row = cw + RSTEP * (vi - i * VPT);
                if (i < T)
                    a.y[(((size_t)b * T + i) * H + h) * P + row] =
                        fmaf(dec[hh * T + i], part[0], rt[(hh * T + i) * P + row]);
            }
            if (pre) {
                // fold the buffered records into this warp's rows (the flush's arithmetic)
                const float *wh = wf + hh * KM;
                const uint16_t *xh = r_x + hh * KM * P;
                for (int idx = lane; idx < ln * VPT; idx += 32) {
                    const int j = idx / VPT, v = idx - j * VPT, row = cw + RSTEP * v;
                    s_wx[j * P + row] = wh[j] * bf16_at(xh, j * P + row);
                }
                __syncwarp();
                unsigned long long acc01[VPT], acc23[VPT];
#pragma unroll
                for (int v = 0; v < VPT; ++v) acc01[v] = acc23[v] = 0ull;
                for (int j = 0; j < ln; ++j) {
                    const uint2 braw = *reinterpret_cast<const uint2 *>(r_B + j * N + col4 * 4);
                    const unsigned long long b01 = f2pack(bf16lo(braw.x), bf16hi(braw.x));
                    const unsigned long long b23 = f2pack(bf16lo(braw.y), bf16hi(braw.y));
#pragma unroll
                    for (int v = 0; v < VPT; ++v) {
                        const float c = s_wx[j * P + cw + RSTEP * v];
                        const unsigned long long cc = f2pack(c, c);
                        acc01[v] = fma2(cc, b01, acc01[v]);
                        acc23[v] = fma2(cc, b23, acc23[v]);
                    }
                }
                const unsigned long long dd = f2pack(fdec[hh], fdec[hh]);
                float4 *ckp = reinterpret_cast<float4 *>(a.ckpt + tile * N);
                float4 o[VPT];
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    f2unpack(fma2(dd, f2pack(hv[v].x, hv[v].y), acc01[v]), o[v].x, o[v].y);
                    f2unpack(fma2(dd, f2pack(hv[v].z, hv[v].w), acc23[v]), o[v].z, o[v].w);
                    st_stream(ckp + ctid + v * NC, o[v]);
                }
                if (a.read_copy == 2) {
                    nv4_quantize_store(o, a.ckpt_q + (tile / P) * nv4_head_bytes(P, N), a.ckpt_scale + tile, P, N,
                                       [&](int v) { return cw + RSTEP * v; });
                } else if (a.read_copy) {
                    uint32_t q[VPT];
                    float rs;
                    e4m3_quantize_rows<VPT>(o, q, rs);
                    uint32_t *ckq = reinterpret_cast<uint32_t *>(a.ckpt_q + tile * N);
#pragma unroll
                    for (int v = 0; v < VPT; ++v) ckq[ctid + v * NC] = q[v];
                    if (reduced_writer<32, VPT>()) a.ckpt_scale[tile + cw + RSTEP * reduced_index<32, VPT>(0)] = rs;
                }
                __syncwarp();                            // s_wx is rewritten for the next head
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (pitem) mbar_arrive(rempty + r);          // record buffer r may be refilled
            mbar_arrive(pempty + ia);                    // and the item arrays ia
        }
    }
    if (ctid == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
}

// After the verify kernel: the drafts' B and C rows (shared by the heads of a
// group) go to the last T slots of each sequence's ring, whose pointers the
// verify kernel has already committed.
__global__ void verify_bc_epilogue(const M2Args a) {
    const int b = blockIdx.x;
    const int sb = a.slots ? a.slots[b] : b;
    if (sb < 0 || sb >= a.cap) return;
    const int hd = a.ring_head[sb], ln = a.ring_len[sb], L = a.L, T = a.T, G = a.G, N = a.N;
    if (hd < 0 || hd >= L || ln < T || ln > L) return;
    const int CB = N / 8;
    const int total = 2 * T * G * CB;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const bool isC = idx >= T * G * CB;
        const int rr = isC ? idx - T * G * CB : idx;
        const int i = rr / (G * CB), r2 = rr - i * G * CB, g = r2 / CB, c = r2 - g * CB;
        uint16_t *dst = static_cast<uint16_t *>(isC ? a.rec_C : a.rec_B);
        if (dst == nullptr) continue;
        const uint16_t *src = static_cast<const uint16_t *>(isC ? a.Cin : a.Bin);
        const int slot = (hd + ln - T + i) % L;
        *reinterpret_cast<uint4 *>(dst + ((((size_t)sb * G + g) * L + slot) * N + c * 8)) =
            __ldcg(reinterpret_cast<const uint4 *>(src + ((((size_t)b * T + i) * G + g) * N + c * 8)));
    }
}

}  // namespace rssm
