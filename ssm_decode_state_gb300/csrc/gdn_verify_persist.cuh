// Persistent, warp-specialised speculative verify of T <= 4 drafts for the
// gated delta rule at the serving head shape (dk = dv = 128, bf16 inputs).
//
// Same pipeline as the persistent decode (gdn_persist.cuh): one CTA per SM
// walks a static list of items, one (sequence, head) each; the state streams
// through shared memory as two 64-row stages.  The records of an item are its
// len buffered ones plus the T drafts; draft i is scored causally, from the
// checkpoint, the buffered records and drafts 1..i:
//   o_i = S_c u_0(i) + sum_{j <= len + i} beta_j (k_j . u_j(i)) v_j,
//   u_{len+i}(i) = q_i, u_{j-1}(i) = alpha_j (u_j(i) - beta_j (k_j . u_j(i)) k_j).
// If len + T > L the buffered records are first folded into the checkpoint
// (the pre-flush, the flush's re-associated arithmetic); the outputs are read
// from the unfolded checkpoint plus every record, which is the same number.
// Drafts are never folded by a verify, so rejecting them stays a pointer move.
//
//  * tile warp: bulk copies of the state halves (as the decode).
//  * record warp: per item, the used ring runs of k and v and every draft's
//    q, k and v rows by bulk copy, alpha and beta by cp.async.
//  * preparation warps, alternate items: append the drafts to the ring, run
//    the T backward chains together (their dot products share one transposed
//    reduction), leave u_0(i) and the record terms of every row, and on a
//    pre-flush the fold constants of the buffered records.  An item without a
//    pre-flush needs nothing more from its record buffer, and the preparation
//    releases it.
//  * consumer warps: per stage, the T dot products of each row with the u_0(i)
//    (one transposed reduction), the outputs, and on a pre-flush the fold.
//
// Ring pointers are read once at kernel start and committed there by the
// sequence's last arrival: pre-flush -> head <- (head + len) mod L, len <- T;
// otherwise len <- len + T.  Every wait is bounded.
#pragma once

#include "gdn_persist.cuh"

namespace rssm {

constexpr int kGdnVT = 4;      // drafts a verify item holds in registers

// Packed float32 pair product (the sm_100 two-wide multiply, each lane rounded
// as a scalar multiply).
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// A bf16 pair (low element first) as a packed float32 pair (exact).
__device__ __forceinline__ unsigned long long bf16x2_to_f2(uint32_t w) {
    return f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Byte layout of the verify kernel's shared memory (KM = L + T records).
struct GVPSmem {
    int stage_bytes, stages_off, full_off, empty_off, rfull_off, rempty_off, pfull_off, pempty_off;
    int rk_off, rv_off, rq_off, ral_off, rbe_off, rec_bytes, rec_off;
    int meta_off, u_off, rt_off, fc_off, f_off, flag_off, total;
    __host__ __device__ GVPSmem(int DK, int DV, int L, int T, int S, int RB, int MY) {
        const int KM = L + T;
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
        // one record buffer: k [KM][DK] bf16, v [KM][DV] bf16, q [T][DK] bf16, alpha, beta [KM] f32
        rk_off = 0;
        rv_off = up(KM * DK * 2, 16);
        rq_off = rv_off + up(KM * DV * 2, 16);
        ral_off = rq_off + up(T * DK * 2, 16);
        rbe_off = ral_off + up(KM * 4, 16);
        rec_bytes = up(rbe_off + KM * 4, 128);
        rec_off = o;  o += RB * rec_bytes;
        meta_off = o; o += up(MY * 12, 16);                       // [items of this CTA][head, len, cache slot]
        u_off = o;    o += up(kGdnBufs * kGdnVT * DK * 4, 16);    // u_0 per draft per prepared item
        rt_off = o;   o += up(kGdnBufs * kGdnVT * DV * 4, 16);    // record term per draft per prepared item
        fc_off = o;   o += up(kGdnBufs * kFcStride * 4, 16);      // pre-flush fold constants per prepared item
        f_off = o;    o += up(8 * kGdnMaxRec * 8 * 4, 16);        // fold coefficients, [warp][j][8 rows]
        flag_off = o; o += 16;
        total = o;
    }
};

template <int DK, int DV>
__global__ void __launch_bounds__(256 + 64 + kPrepThreads, 1) gdn_verify_persistent(const GPArgs a) {
    constexpr int NC = 256, VPT = 8, G4 = DK / 4, RSTEP = NC / G4, NU = DV / kGdnRows, TQ = kGdnVT;
    static_assert(G4 == 32 && NC * VPT * 4 == kGdnRows * DK && DV % kGdnRows == 0, "serving shape");
    static_assert(TQ * VPT == 32, "one (draft, row) pair per lane after the reduction");
    constexpr int CK = DK / 8, CV = DV / 8;              // 16-byte chunks per k / v row
    extern __shared__ __align__(128) unsigned char smraw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.L, H = a.H, S = a.stages, RB = a.recbufs, T = a.T;
    const GVPSmem lay(DK, DV, L, T, S, RB, a.max_my);
    unsigned char *stages = smraw + lay.stages_off;
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + lay.full_off);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smraw + lay.empty_off);
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smraw + lay.rfull_off);
    uint64_t *rempty = reinterpret_cast<uint64_t *>(smraw + lay.rempty_off);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smraw + lay.pfull_off);
    uint64_t *pempty = reinterpret_cast<uint64_t *>(smraw + lay.pempty_off);
    int *s_meta = reinterpret_cast<int *>(smraw + lay.meta_off);
    float *s_u = reinterpret_cast<float *>(smraw + lay.u_off);
    float *s_rt = reinterpret_cast<float *>(smraw + lay.rt_off);
    float *s_fc = reinterpret_cast<float *>(smraw + lay.fc_off);
    float *s_f = reinterpret_cast<float *>(smraw + lay.f_off);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smraw + lay.flag_off);

    const int grid = gridDim.x;
    const int n_my = (a.items - (int)blockIdx.x + grid - 1) / grid;
    auto item_of = [&](int k) { return (int)blockIdx.x + k * grid; };   // item = b * H + h
    auto meta_bad = [&](int hd, int ln) { return hd < 0 || hd >= L || ln < 0 || ln > L; };
    // an item that pre-flushes: its consumers fold its buffered records (read from the
    // record buffer) and release that buffer; every other buffer the preparation releases
    auto pre_item = [&](int hd, int ln) { return !meta_bad(hd, ln) && ln + T > L; };
    auto rec = [&](int r) { return smraw + lay.rec_off + r * lay.rec_bytes; };
    auto cb_of = [&](int k) { return (size_t)s_meta[k * 3 + 2] * H + (size_t)(item_of(k) % H); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, NC / 32);
        }
        for (int r = 0; r < RB; ++r) {
            mbar_init(rfull + r, 33);                    // 32 cp.async arrivals + lane 0's
            mbar_init(rempty + r, NC / 32);
        }
        for (int i = 0; i < kGdnBufs; ++i) {
            mbar_init(pfull + i, 1);
            mbar_init(pempty + i, NC / 32);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    for (int k = tid; k < n_my; k += blockDim.x) {
        const int it = item_of(k), b = it / H;
        const int sb = a.slots ? __ldg(a.slots + b) : b;
        if (sb < 0 || sb >= a.cap) {
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
            const size_t cbh = cb_of(k);
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
            *s_abort = 1;
            flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        }
        // the copies in flight land before the CTA ends (see the decode's tile warp)
        for (int u = issued - S < 0 ? 0 : issued - S; u < issued; ++u)
            mbar_wait(full + (u % S), (uint32_t)((u / S) & 1));
        return;
    }

    if (warp == 1) {
        // ================================ record warp =================================
        bool ok = true;
        int k = 0;
        for (; k < n_my; ++k) {
            const int r = k % RB;
            if (lane == 0 && k >= RB) ok = pwait(rempty + r, (uint32_t)(((k / RB) - 1) & 1), s_abort) && !*s_abort;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const int it = item_of(k), b = it / H, h = it - b * H;
            const size_t cbh = cb_of(k);
            const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1];
            const bool good = !meta_bad(hd, ln);
            if (good) {
                // records: list position j < ln is ring slot (hd + j) mod L, j = ln + i draft i
                unsigned char *rb = rec(r);
                const int run1 = ln < L - hd ? ln : L - hd, run2 = ln - run1;
                if (lane == 0)
                    mbar_arrive_expect_tx(rfull + r, (uint32_t)(((ln + T) * (DK + DV) + T * DK) * 2));
                __syncwarp();
                if (lane == 0) {
                    unsigned char *d = rb + lay.rk_off;
                    if (run1) bulk_g2s(d, a.rec_k + (cbh * L + hd) * DK, run1 * DK * 2, rfull + r);
                    if (run2) bulk_g2s(d + run1 * DK * 2, a.rec_k + cbh * L * DK, run2 * DK * 2, rfull + r);
                } else if (lane == 1) {
                    unsigned char *d = rb + lay.rv_off;
                    if (run1) bulk_g2s(d, a.rec_v + (cbh * L + hd) * DV, run1 * DV * 2, rfull + r);
                    if (run2) bulk_g2s(d + run1 * DV * 2, a.rec_v + cbh * L * DV, run2 * DV * 2, rfull + r);
                } else if (lane >= 2 && lane < 2 + 3 * T) {
                    // draft i's k, v and q rows: inputs [b][T][H][d]
                    const int w = lane - 2, i = w / 3, which = w - 3 * i;
                    const size_t src = ((size_t)b * T + i) * H + h;
                    if (which == 0)
                        bulk_g2s(rb + lay.rk_off + (ln + i) * DK * 2, a.k + src * DK, DK * 2, rfull + r);
                    else if (which == 1)
                        bulk_g2s(rb + lay.rv_off + (ln + i) * DV * 2, a.v + src * DV, DV * 2, rfull + r);
                    else
                        bulk_g2s(rb + lay.rq_off + i * DK * 2, a.q + src * DK, DK * 2, rfull + r);
                }
                for (int j = lane; j < ln + T; j += 32) {
                    const int slot = hd + j < L ? hd + j : hd + j - L;
                    const size_t dsrc = ((size_t)b * T + (j - ln)) * H + h;
                    cp_async4(rb + lay.ral_off + j * 4, j < ln ? a.rec_alpha + cbh * L + slot : a.alpha + dsrc);
                    cp_async4(rb + lay.rbe_off + j * 4, j < ln ? a.rec_beta + cbh * L + slot : a.beta + dsrc);
                }
            }
            cp_async_arrive_noinc(rfull + r);
            if (lane == 0 && !good) mbar_arrive(rfull + r);
        }
        cp_async_wait_all();
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
        const int pw = warp - 2 - NC / 32;               // 0 or 1: even or odd items
        bool live = true;
        for (int kk = pw; kk < n_my; kk += 2) {
            const int r = kk % RB, ib = kk % kGdnBufs;
            if (live && kk >= kGdnBufs && !pwait(pempty + ib, (uint32_t)(((kk / kGdnBufs) - 1) & 1), s_abort)) {
                live = false;
                *s_abort = 1;
            }
            if (live && !pwait(rfull + r, (uint32_t)((kk / RB) & 1), s_abort)) {
                live = false;
                *s_abort = 1;
            }
            const size_t cbh = cb_of(kk);
            const int hd = s_meta[kk * 3 + 0], ln = s_meta[kk * 3 + 1];
            const bool work = live && !meta_bad(hd, ln);
            const bool pre = ln + T > L;
            const unsigned char *rb = rec(r);
            const uint16_t *r_k = reinterpret_cast<const uint16_t *>(rb + lay.rk_off);
            const uint16_t *r_v = reinterpret_cast<const uint16_t *>(rb + lay.rv_off);
            const uint16_t *r_q = reinterpret_cast<const uint16_t *>(rb + lay.rq_off);
            const float *r_al = reinterpret_cast<const float *>(rb + lay.ral_off);
            const float *r_be = reinterpret_cast<const float *>(rb + lay.rbe_off);
            // the drafts' rows for the ring, read now (the record buffer may be handed back
            // below) and stored after the hand-over, so that no release waits for them
            constexpr int NA = kGdnVT * (CK + CV) / 32;  // 16-byte chunks per lane
            uint4 app[NA];
            if (work) {
#pragma unroll
                for (int q = 0; q < NA; ++q) {
                    const int idx = lane + 32 * q, i = idx / (CK + CV), c = idx - i * (CK + CV);
                    app[q] = i < T ? (c < CK ? *reinterpret_cast<const uint4 *>(r_k + (ln + i) * DK + c * 8)
                                             : *reinterpret_cast<const uint4 *>(r_v + (ln + i) * DV + (c - CK) * 8))
                                   : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            const float app_al = (work && lane < T) ? r_al[ln + lane] : 0.0f;
            const float app_be = (work && lane < T) ? r_be[ln + lane] : 0.0f;
            if (work) {
                // the T backward chains, newest record first; chain i starts at record ln + i.
                // Lane (i, c) = (lane / 8, lane % 8) runs chain i on columns 16 c .. 16 c + 15
                // of u(i) and rows 16 c .. 16 c + 15 of its record term: a step's dot product
                // reduces over the chain's 8 lanes (3 shuffle levels).
                const int ci = lane >> 3, c8 = lane & 7;
                // packed float32 pairs (columns / rows 2m, 2m + 1 of the lane's 16): the
                // sm_100 two-wide fma, mul and add, each lane of a pair rounded as a scalar op
                unsigned long long u2[8], racc2[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    u2[m] = ci < T ? bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(r_q + ci * DK + 16 * c8 + 2 * m))
                                   : 0ull;
                    racc2[m] = 0ull;
                }
                for (int j = ln + T - 1; j >= 0; --j) {
                    const uint4 k0 = *reinterpret_cast<const uint4 *>(r_k + j * DK + 16 * c8);
                    const uint4 k1 = *reinterpret_cast<const uint4 *>(r_k + j * DK + 16 * c8 + 8);
                    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                    unsigned long long kj2[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) kj2[m] = bf16x2_to_f2(kw[m]);
                    unsigned long long pa = 0ull, pb = 0ull;
#pragma unroll
                    for (int m = 0; m < 8; m += 2) {
                        pa = fma2(kj2[m], u2[m], pa);
                        pb = fma2(kj2[m + 1], u2[m + 1], pb);
                    }
                    float d0, d1, d2, d3;
                    f2unpack(pa, d0, d1);
                    f2unpack(pb, d2, d3);
                    float d = (d0 + d2) + (d1 + d3);
                    d += __shfl_xor_sync(0xffffffffu, d, 1);
                    d += __shfl_xor_sync(0xffffffffu, d, 2);
                    d += __shfl_xor_sync(0xffffffffu, d, 4);
                    if (ci < T && j <= ln + ci) {                // chain ci has reached record j
                        const float cf = r_be[j] * d, al = r_al[j];
                        const unsigned long long cf2 = f2pack(cf, cf), ncf2 = f2pack(-cf, -cf), al2 = f2pack(al, al);
                        const uint4 v0 = *reinterpret_cast<const uint4 *>(r_v + j * DV + 16 * c8);
                        const uint4 v1 = *reinterpret_cast<const uint4 *>(r_v + j * DV + 16 * c8 + 8);
                        const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                        for (int m = 0; m < 8; ++m) {
                            racc2[m] = fma2(cf2, bf16x2_to_f2(vw[m]), racc2[m]);
                            u2[m] = mul2(al2, fma2(ncf2, kj2[m], u2[m]));
                        }
                    }
                }
                float4 *su = reinterpret_cast<float4 *>(s_u + (ib * TQ + ci) * DK + 16 * c8);
                float4 *sr = reinterpret_cast<float4 *>(s_rt + (ib * TQ + ci) * DV + 16 * c8);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float a0, a1, a2, a3, b0, b1, b2, b3;
                    f2unpack(u2[2 * m], a0, a1);
                    f2unpack(u2[2 * m + 1], a2, a3);
                    f2unpack(racc2[2 * m], b0, b1);
                    f2unpack(racc2[2 * m + 1], b2, b3);
                    su[m] = make_float4(a0, a1, a2, a3);
                    sr[m] = make_float4(b0, b1, b2, b3);
                }
                if (pre) gdn_fold_constants<DK>(s_fc + ib * kFcStride, r_k, r_al, ln);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(pfull + ib);                 // item kk is prepared
                if (!pre_item(hd, ln)) mbar_arrive_n(rempty + r, NC / 32);
            }
            if (work) {
                // the drafts go to ring slots (hd2 + ln2 + i) mod L, after the pre-flush's
                // pointer move; the ring's old contents were copied before this launch's
                // preparation of the item, and no one reads these slots during the launch
                const int hd2 = pre ? (hd + ln) % L : hd, ln2 = pre ? 0 : ln;
#pragma unroll
                for (int q = 0; q < NA; ++q) {
                    const int idx = lane + 32 * q, i = idx / (CK + CV), c = idx - i * (CK + CV);
                    if (i < T) {
                        const int slot = (hd2 + ln2 + i) % L;
                        if (c < CK)
                            *reinterpret_cast<uint4 *>(a.rec_k + (cbh * L + slot) * DK + c * 8) = app[q];
                        else
                            *reinterpret_cast<uint4 *>(a.rec_v + (cbh * L + slot) * DV + (c - CK) * 8) = app[q];
                    }
                }
                if (lane < T) {
                    const int slot = (hd2 + ln2 + lane) % L;
                    a.rec_alpha[cbh * L + slot] = app_al;
                    a.rec_beta[cbh * L + slot] = app_be;
                }
            }
        }
        if (lane == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
        return;
    }

    // ================================ consumer warps =================================
    const int ctid = tid - 64;                           // 0..255
    const int cw = ctid >> 5;                            // owns rows cw + RSTEP * v of each stage
    const int col4 = lane;
    bool live = true;
    int u = 0;
    for (int k = 0; k < n_my; ++k) {
        const int r = k % RB, ib = k % kGdnBufs;
        const int it = item_of(k), b = it / H, h = it - b * H;
        const size_t cbh = cb_of(k);
        const int hd = s_meta[k * 3 + 0], ln = s_meta[k * 3 + 1];
        const bool pitem = pre_item(hd, ln);
        if (live && !pwait(pfull + ib, (uint32_t)((k / kGdnBufs) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        if (pitem && live && !pwait(rfull + r, (uint32_t)((k / RB) & 1), s_abort)) {
            live = false;
            *s_abort = 1;
        }
        const bool work = live && !meta_bad(hd, ln);
        const bool pre = work && pitem;
        const unsigned char *rb = rec(r);
        const uint16_t *r_k = reinterpret_cast<const uint16_t *>(rb + lay.rk_off);
        const uint16_t *r_v = reinterpret_cast<const uint16_t *>(rb + lay.rv_off);
        const float *r_al = reinterpret_cast<const float *>(rb + lay.ral_off);
        const float *r_be = reinterpret_cast<const float *>(rb + lay.rbe_off);
        float4 u0[TQ];
#pragma unroll
        for (int i = 0; i < TQ; ++i) u0[i] = *reinterpret_cast<const float4 *>(s_u + (ib * TQ + i) * DK + col4 * 4);
        const float *rt = s_rt + ib * TQ * DV;
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
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
            if (!work) continue;
            // o_i = S_c . u_0(i) + record term: the T x 8 row dot products, one
            // transposed reduction; lane ends with (draft, row)
            float part[TQ * VPT];
#pragma unroll
            for (int i = 0; i < TQ; ++i) {
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    float d = hv[v].x * u0[i].x;
                    d = fmaf(hv[v].y, u0[i].y, d);
                    d = fmaf(hv[v].z, u0[i].z, d);
                    d = fmaf(hv[v].w, u0[i].w, d);
                    part[i * VPT + v] = d;
                }
            }
            group_reduce<G4, TQ * VPT>(part);
            {
                const int vi = reduced_index<G4, TQ * VPT>(0);
                const int i = vi / VPT, row = uu * kGdnRows + cw + RSTEP * (vi - i * VPT);
                if (i < T) a.o[(((size_t)b * T + i) * H + h) * DV + row] = part[0] + rt[i * DV + row];
            }
            if (pre)
                gdn_fold_stage<DK, DV, VPT>(hv, ln, r_k, r_v, r_al, r_be, s_fc + ib * kFcStride,
                                            s_f + cw * (kGdnMaxRec * 8), uu, cw,
                                            reinterpret_cast<float4 *>(a.ckpt + (cbh * DV + uu * kGdnRows) * DK));
        }
        __syncwarp();
        if (lane == 0) {
            if (pitem) mbar_arrive(rempty + r);          // record buffer r may be refilled
            mbar_arrive(pempty + ib);
        }
    }
    if (ctid == 0 && !live) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
}

}  // namespace rssm
