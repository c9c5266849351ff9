// Single-pass Mamba-2 replay decode for small batches (serving shape: headdim 64,
// dstate 128, bf16 token inputs, float32 checkpoint without a read copy).
//
// At a few sequences the whole state sits in L2 and a decode step is bound by
// chains of dependent latencies, not by HBM: the persistent kernel's hand-overs
// (ring pointers, then records, then the item's preparation, then the tiles) each
// wait on the one before, and with about one item per SM nothing hides them.
// Here the checkpoint copy starts at once and the warps meet three times:
//
//  * one CTA per (sequence, head): 8 compute warps of 8 checkpoint rows each
//    (lane = 4 columns, as the persistent kernel's consumers) and one
//    bookkeeping warp;
//  * the compute warps load C_t and copy the checkpoint tile into shared memory,
//    each warp its own 8 rows by one bulk copy (the TMA engine) completing on the
//    warp's own mbarrier;
//  * the bookkeeping warp reads the ring pointers and hands them over (first
//    barrier); the compute warps then copy the used ring slots' B and x rows in
//    list order, B_t and x_t last, each lane the B chunks it multiplies with C_t
//    itself, and form B_j . C_t per list position as soon as their own copies
//    have landed;
//  * meanwhile the bookkeeping warp arrives on the sequence's counter (the last
//    of the sequence's H arrivals commits the new pointers: every CTA of the
//    sequence has read the old ones by then), forms the suffix sums S_j (dt of
//    the newer records, newest first), w_j = exp(A S_j) dt_j and exp(A S), hands
//    them over (second barrier), and appends the token to the ring on non-flush
//    steps;
//  * each warp forms h_c . C_t of its rows as soon as it finds them landed: while
//    the records are still on their way (small batches), or else after the lane
//    that holds a row's product has formed the row's record term
//    sum_j w_j (B_j . C_t) x_j + D x_t, so that at most that product follows the
//    tile's arrival; then y = exp(A S) (h_c . C_t) + record term; a flush step
//    (after a third barrier, among the compute warps) folds
//    h_c <- exp(A S) h_c + sum_j w_j x_j B_j^T from the tile in shared memory and
//    stores it.
//
// Each sum is formed with the persistent kernel's operations in its order (the
// same 16-column pair products and butterfly for B_j . C_t, the same newest-first
// suffix sums, the same per-row chains of fused multiply-adds, the same
// cross-lane reduction of h_c . C_t, the same packed fold), so the two kernels
// give the same bits for a sequence and a caller can switch between them with
// the batch size.  The checkpoint is read and written with the default L2
// policy: at these batches it stays resident from one step to the next.
#include <atomic>

#include "common.cuh"
#include "host_common.h"
#include "mamba2_replay.cuh"
#include "persist_common.cuh"

namespace rssm {
namespace {

constexpr int kSmallP = 64, kSmallN = 128;
constexpr int kSmallCompute = kSmallP / 8 * 32;          // 8 warps of 8 rows
constexpr int kSmallThreads = kSmallCompute + 32;        // + the bookkeeping warp

// Named barriers: 1 among the compute warps; 2 and 3 between them and the
// bookkeeping warp (the compute warps wait, the bookkeeping warp only arrives):
// 2 hands over the ring pointers, 3 the decay weights.
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kSmallCompute) : "memory");
}
template <int ID>
__device__ __forceinline__ void handover_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(kSmallThreads) : "memory");
}
template <int ID>
__device__ __forceinline__ void handover_arrive() {
    asm volatile("bar.arrive %0, %1;" ::"n"(ID), "n"(kSmallThreads) : "memory");
}

__global__ void __launch_bounds__(kSmallThreads, 4) m2_decode_small(const M2Args a) {
    constexpr int N = kSmallN, P = kSmallP, VPT = 8, G4 = N / 4, KMX = kMaxL + 1;
    constexpr int CX = P / 8, CB = N / 8;                // 16-byte chunks per x / B row
    extern __shared__ __align__(16) float4 s_h[];        // the checkpoint tile [P][N / 4]
    // the records by list position j = 0..ln (the ring slots in order, then the
    // current token): B rows of the group, x rows of the head
    __shared__ __align__(16) uint16_t s_rB[KMX * N];
    __shared__ __align__(16) uint16_t s_rx[KMX * P];
    __shared__ __align__(16) float s_w[KMX], s_cbs[KMX];
    __shared__ __align__(16) float s_wx[KMX * P];        // flush: w_j x_j per row
    __shared__ uint64_t s_bar[kSmallCompute / 32];      // per compute warp: its tile rows landed
    __shared__ int s_meta[2];
    __shared__ float s_dec;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y;
    const int H = a.H, G = a.G, L = a.L, g = h / a.hpg;
    const int sb = a.slots ? __ldg(a.slots + b) : b;     // the sequence's cache slot
    if (sb < 0 || sb >= a.cap) {
        if (h == 0 && tid == 0) flag_error(a.err, RSSM_DEVERR_SLOT);
        return;
    }
    const size_t bh = (size_t)sb * H + h, bg = (size_t)sb * G + g;

    if (warp == kSmallCompute / 32) {
        // =============================== bookkeeping warp ===============================
        // The ring pointers, the head's dt ring (lane = slot), the current dt and A, and
        // the token's record for the append, all in one round trip.
        const int hd = __ldcg(a.ring_head + sb), ln = __ldcg(a.ring_len + sb);
        const float rdt = lane < L ? __ldcg(a.rec_dt + bh * L + lane) : 0.0f;
        const float dtt = __ldcg(a.dt + (size_t)b * H + h), Ah = __ldg(a.A + h);
        const bool good = hd >= 0 && hd < L && ln >= 0 && ln <= L;
        const bool fold = ln + 1 >= L;
        const int nBC = (h % a.hpg == 0) ? 2 * CB : 0;       // the group's first head writes B and C
        const int nap = (good && !fold) ? CX + nBC : 0;      // 16-byte chunks to append
        uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
        auto chunk_src = [&](int idx) -> const uint4 * {
            if (idx < CX)
                return reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.x) + ((size_t)b * H + h) * P) + idx;
            const int rr = idx - CX;
            const bool isC = rr >= CB;
            return reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(isC ? a.Cin : a.Bin) +
                                                   ((size_t)b * G + g) * N) + (isC ? rr - CB : rr);
        };
        // the token's chunks are loaded whatever the pointers say (no wait on them);
        // only nap of them are stored
        if (lane < CX + nBC) v0 = __ldcg(chunk_src(lane));
        if (lane + 32 < CX + nBC) v1 = __ldcg(chunk_src(lane + 32));
        if (lane == 0) {
            s_meta[0] = hd;
            s_meta[1] = ln;
        }
        __syncwarp();
        handover_arrive<2>();                            // the pointers
        // Arrive on the sequence's counter as soon as the pointers are in; the result
        // is needed only after the weights, so the round trip overlaps them.
        // Ordering without fences: the arrival depends on the loaded pointer values
        // (it is issued only for good ones), so it leaves after they have returned;
        // the commit depends on the last arrival's result, so it leaves after every
        // CTA of the sequence has arrived, i.e. after every read of the old pointers.
        // The atomic is predicated, not branched around: a branch would merge its
        // result at the reconvergence point and hold the warp for the round trip.
        int prior = -1;
        {
            const uint32_t on = (good && lane == 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p atom.global.add.u32 %0, [%1], 1;\n\t}"
                : "+r"(prior)
                : "l"(a.arrive + sb), "r"(on)
                : "memory");
        }
        if (good) {
            // dt in list order (position j < ln is slot (hd + j) mod L, position ln the
            // current token): lane j takes position j's value; position 32 (ln = 32)
            // is dt_t, the newest
            const int sl = lane < ln ? (hd + lane < L ? hd + lane : hd + lane - L) : 0;
            const float dsl = __shfl_sync(0xffffffffu, rdt, sl);
            const float dpos = lane < ln ? dsl : dtt;
            // suffix sums, newest first (lane j: the positions after j) and the total.
            // Every position is broadcast in turn; the loop is unrolled so that the
            // broadcasts issue back to back and only the adds form a chain
            float sf = 0.0f, tot = 0.0f;
            if (ln == 32) {
                sf = dtt;
                tot = dtt;
            }
#pragma unroll
            for (int i = 31; i >= 0; --i) {
                const float di = __shfl_sync(0xffffffffu, dpos, i);
                if (i <= ln) {
                    if (i > lane) sf += di;
                    tot += di;
                }
            }
            // w_j = exp(A S_j) dt_j and exp(A S)
            if (lane <= ln) s_w[lane] = expf(Ah * sf) * dpos;
            if (lane == 0 && ln == 32) s_w[32] = expf(Ah * 0.0f) * dtt;
            if (lane == 0) s_dec = expf(Ah * tot);
        }
        __syncwarp();
        handover_arrive<3>();                            // w and exp(A S)
        if (!good) {
            if (h == 0 && lane == 0) flag_error(a.err, RSSM_DEVERR_RING_META);
            return;
        }
        if (lane == 0 && prior == H - 1) {
            // the sequence's last arrival commits the new pointers
            a.ring_head[sb] = fold ? (hd + ln + 1) % L : hd;
            a.ring_len[sb] = fold ? 0 : ln + 1;
            a.arrive[sb] = 0;
        }
        if (nap) {
            // the token goes to slot (hd + ln) mod L, which no CTA reads for this step
            const int slot = hd + ln < L ? hd + ln : hd + ln - L;
            auto chunk_dst = [&](int idx) -> uint4 * {
                if (idx < CX)
                    return reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.rec_x) + (bh * L + slot) * P) + idx;
                const int rr = idx - CX;
                const bool isC = rr >= CB;
                uint16_t *base = static_cast<uint16_t *>(isC ? a.rec_C : a.rec_B);
                return base ? reinterpret_cast<uint4 *>(base + (bg * L + slot) * N) + (isC ? rr - CB : rr) : nullptr;
            };
            if (lane < nap) {
                uint4 *d = chunk_dst(lane);
                if (d) *d = v0;
            }
            if (lane + 32 < nap) {
                uint4 *d = chunk_dst(lane + 32);
                if (d) *d = v1;
            }
            if (lane == 0) a.rec_dt[bh * L + slot] = dtt;
        }
        return;
    }

    // ================================ compute warps ==================================
    const int cw = warp;                                 // owns rows cw * 8 .. cw * 8 + 7
    const float Dh = __ldg(a.D + h);
    // C_t first (it gates both products below): this lane's 4 columns of the row
    // dot products and its 16 columns of B . C, through L1 (every warp of the CTA
    // reads the same 256 bytes)
    const int c0 = (lane & 7) * 16;                      // this lane's B / C columns
    const uint16_t *gC = static_cast<const uint16_t *>(a.Cin) + ((size_t)b * G + g) * N;
    const uint2 craw = __ldg(reinterpret_cast<const uint2 *>(gC) + lane);
    const uint4 q0 = __ldg(reinterpret_cast<const uint4 *>(gC + c0));
    const uint4 q1 = __ldg(reinterpret_cast<const uint4 *>(gC + c0 + 8));
    // The warp's 8 rows of the tile (4 KiB) by one bulk copy on the warp's own
    // mbarrier: their arrival is tracked apart from the record copies below, so
    // that everything but h_c . C_t is formed while the tile is still arriving.
    const float4 *ck = reinterpret_cast<const float4 *>(a.ckpt) + bh * P * G4;
    uint64_t *bar = s_bar + cw;
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, VPT * G4 * 16);
        bulk_g2s(s_h + cw * VPT * G4, ck + cw * VPT * G4, VPT * G4 * 16, bar);
    }
    __syncwarp();
    // A bounded wait for the warp's rows; if it gives up (flagged), wait once more
    // so that the copy has landed before the CTA can end, and store nothing.
    bool lost = false;
    auto wait_tile = [&]() {
        if (!mbar_wait(bar, 0)) {
            lost = true;
            if (lane == 0) flag_error(a.err, RSSM_DEVERR_TIMEOUT);
            mbar_wait(bar, 0);
        }
    };
    // Two groups of record copies, each thread its own share: (0) the B chunks this
    // lane multiplies with C_t below (8 lanes per list position, 16 columns per
    // lane, 4 positions per warp and pass), (1) x rows, read by other threads after
    // the last hand-over.
    handover_sync<2>();                                  // the ring pointers
    const int hd = s_meta[0], ln = s_meta[1];
    const bool bad = hd < 0 || hd >= L || ln < 0 || ln > L;   // flagged by the bookkeeping warp
    const int nrec = bad ? 0 : ln + 1;                   // list positions to stage
    // ring slot of list position j < ln; position ln is the current token
    auto slot_of = [&](int j) { return hd + j < L ? hd + j : hd + j - L; };
    {
        const uint16_t *gB = static_cast<const uint16_t *>(a.rec_B) + bg * L * N;
        const uint16_t *gBt = static_cast<const uint16_t *>(a.Bin) + ((size_t)b * G + g) * N;
        for (int jb = 4 * cw; jb < nrec; jb += 4 * (kSmallCompute / 32)) {
            const int j = jb + (lane >> 3);
            if (j < nrec) {
                const uint16_t *src = (j < ln ? gB + slot_of(j) * N : gBt) + c0;
                cp_async16(s_rB + j * N + c0, src);
                cp_async16(s_rB + j * N + c0 + 8, src + 8);
            }
        }
    }
    cp_async_commit();
    {
        const uint16_t *gx = static_cast<const uint16_t *>(a.rec_x) + bh * L * P;
        const uint16_t *gxt = static_cast<const uint16_t *>(a.x) + ((size_t)b * H + h) * P;
        for (int idx = tid; idx < nrec * CX; idx += kSmallCompute) {
            const int j = idx / CX, c = idx - j * CX;
            cp_async16(s_rx + j * P + c * 8, (j < ln ? gx + slot_of(j) * P : gxt) + c * 8);
        }
    }
    cp_async_commit();
    cp_async_wait_group<1>();                            // this lane's B chunks
    // B_j . C_t per list position: 16 columns per lane as bf16 pairs, then a
    // 3-level butterfly
    for (int jb = 4 * cw; jb < nrec; jb += 4 * (kSmallCompute / 32)) {
        const int j = jb + (lane >> 3);
        float acc = 0.0f;
        if (j < nrec) {
            const uint4 b0 = *reinterpret_cast<const uint4 *>(s_rB + j * N + c0);
            const uint4 b1 = *reinterpret_cast<const uint4 *>(s_rB + j * N + c0 + 8);
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
        if (j < nrec && (lane & 7) == 0) s_cbs[j] = acc;
    }
    // h_c . C_t of the warp's 8 rows: the writer lane of each row keeps its sum
    const bool writer = reduced_writer<G4, VPT>();
    const int row = cw * VPT + reduced_index<G4, VPT>(0);
    const float4 cfr = make_float4(bf16lo(craw.x), bf16hi(craw.x), bf16lo(craw.y), bf16hi(craw.y));
    float hc = 0.0f;
    auto row_dots = [&]() {
        float part[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const float4 hv = s_h[(cw * VPT + v) * G4 + lane];
            float d = hv.x * cfr.x;
            d = fmaf(hv.y, cfr.y, d);
            d = fmaf(hv.z, cfr.z, d);
            d = fmaf(hv.w, cfr.w, d);
            part[v] = d;
        }
        group_reduce<G4, VPT>(part);
        hc = part[0];
    };
    // if the warp's tile rows are already in (small batches), form their products
    // now, while the records and the weights are still on their way
    const bool early = __shfl_sync(0xffffffffu, mbar_try_wait(bar, 0) ? 1 : 0, 0) != 0;
    if (early) row_dots();
    cp_async_wait_all();
    handover_sync<3>();                                  // records staged; w and exp(A S) known
    if (bad) {
        if (!early) wait_tile();
        return;
    }
    const bool fold = ln + 1 >= L;
    const float dec = s_dec;
    // The lanes that hold a row's h_c . C_t form that row's record term,
    // sum_j w_j (B_j . C_t) x_j + D x_t, while the tile may still be arriving.
    float rt = 0.0f;
    if (writer) {
        float acc = 0.0f;
#pragma unroll 4
        for (int j = 0; j < nrec; ++j) acc = fmaf(s_w[j] * s_cbs[j], bf16_at(s_rx + j * P, row), acc);
        rt = fmaf(Dh, bf16_at(s_rx + ln * P, row), acc);
    }
    if (!early) {
        wait_tile();
        row_dots();
    }
    if (writer && !lost) a.y[((size_t)b * H + h) * P + row] = fmaf(dec, hc, rt);
    if (!fold) return;

    // flush: w_j x_j for every row, then the rank-nrec update and the decayed
    // checkpoint in one fma per element (the state is rounded once per flush)
    for (int idx = tid; idx < nrec * P; idx += kSmallCompute) {
        const int j = idx / P, row = idx - j * P;
        s_wx[idx] = s_w[j] * bf16_at(s_rx + j * P, row);
    }
    compute_sync();
    // four rows at a time (half the accumulators of the warp's 8 rows live at once)
    const unsigned long long dd = f2pack(dec, dec);
    float4 *cko = reinterpret_cast<float4 *>(a.ckpt) + bh * P * G4;
    for (int q = cw * VPT; q < cw * VPT + VPT; q += 4) {
        unsigned long long acc01[4], acc23[4];           // packed (x, y) and (z, w)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc01[v] = acc23[v] = 0ull;
        for (int j = 0; j < nrec; ++j) {
            const uint2 braw = *reinterpret_cast<const uint2 *>(s_rB + j * N + lane * 4);
            const unsigned long long b01 = f2pack(bf16lo(braw.x), bf16hi(braw.x));
            const unsigned long long b23 = f2pack(bf16lo(braw.y), bf16hi(braw.y));
            const float4 wa = *reinterpret_cast<const float4 *>(s_wx + j * P + q);
            const float wv[4] = {wa.x, wa.y, wa.z, wa.w};
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const unsigned long long cc = f2pack(wv[v], wv[v]);
                acc01[v] = fma2(cc, b01, acc01[v]);
                acc23[v] = fma2(cc, b23, acc23[v]);
            }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int e = (q + v) * G4 + lane;
            const float4 hv = s_h[e];
            float4 o;
            f2unpack(fma2(dd, f2pack(hv.x, hv.y), acc01[v]), o.x, o.y);
            f2unpack(fma2(dd, f2pack(hv.z, hv.w), acc23[v]), o.z, o.w);
            if (!lost) __stcg(cko + e, o);
        }
    }
}

}  // namespace

// Batches up to this many sequences take the single-pass kernel: measured (us per
// step, CUDA graphs of 64 steps, this kernel / the persistent kernel) at batch 8
// 8.2 / 12.6, 16 14.4 / 18.2, 32 33.1 / 28.9.
constexpr int kSmallBatchMax = 16;

// Returns RSSM_ERR_UNSUPPORTED (without launching) when the call is not one this
// kernel handles: another shape, a read copy, an FP16 checkpoint, or a batch
// above kSmallBatchMax.
rssm_status launch_decode_small(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st) {
    if (!d->io_bf16 || d->dstate != kSmallN || d->headdim != kSmallP || d->read_copy || d->ckpt_f16)
        return RSSM_ERR_UNSUPPORTED;
    if (d->batch > kSmallBatchMax || d->L > kMaxL) return RSSM_ERR_UNSUPPORTED;
    const size_t smem = (size_t)kSmallP * kSmallN * sizeof(float);     // the checkpoint tile
    // static (~22 KB) + dynamic shared memory is above the 48 KB a block gets
    // without opting in: raise the dynamic limit once per device
    static std::atomic<bool> opted[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RSSM_ERR_CUDA;
    if (!opted[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute((const void *)m2_decode_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return RSSM_ERR_CUDA;
        opted[dev].store(true, std::memory_order_release);
    }
    M2Args a = args;
    void *params[] = {&a};
    if (cudaLaunchKernel((const void *)m2_decode_small, dim3(d->nheads, d->batch), dim3(kSmallThreads), params, smem,
                         st) != cudaSuccess)
        return RSSM_ERR_CUDA;
    return launch_status();
}

}  // namespace rssm
