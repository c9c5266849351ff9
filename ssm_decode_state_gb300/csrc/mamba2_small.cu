// Single-pass Mamba-2 replay decode for small batches (serving shape: headdim 64,
// dstate 128, bf16 token inputs, float32 checkpoint without a read copy).
//
// At a few sequences the whole state sits in L2 and a decode step is bound by
// its chain of dependent latencies, not by bytes: the persistent kernel's
// hand-overs (ring pointers, then records, then the item's preparation, then the
// tiles) each wait on the one before, and with about one item per SM nothing
// hides them.  Here every load of a step is issued at once, and the compute warps
// meet twice at a barrier:
//
//  * one CTA per (sequence, head): 8 compute warps of 8 checkpoint rows each
//    (lane = 4 columns, as the persistent kernel's consumers) and one
//    bookkeeping warp;
//  * the compute warps copy the checkpoint tile into shared memory by cp.async,
//    each thread the elements it reads itself, and each lane the chunks of the
//    group's B ring (every slot: no copy waits for the ring pointers) and of B_t
//    that it multiplies with C_t itself, so that h_c . C_t per row and B_r . C_t
//    per ring slot r are formed as soon as a thread's own copies have landed,
//    with no barrier; the head's x ring and x_t are copied alongside;
//  * meanwhile the bookkeeping warp reads the ring pointers and the head's dt
//    ring, forms the suffix sums S_j (dt of the newer records, newest first),
//    w_j = exp(A S_j) dt_j and exp(A S), and hands them to the compute warps at
//    the one barrier they share with it; then it arrives on the sequence's
//    counter (the last of the sequence's H arrivals commits the new pointers:
//    every CTA of the sequence has read the old ones by then) and appends the
//    token to the ring on non-flush steps;
//  * after that barrier one thread per row forms the record term
//    sum_j w_j (B_j . C_t) x_j + D x_t, taking B_j . C_t from the slot list
//    position j maps to, and y = exp(A S) (h_c . C_t) + record term; a flush step
//    (after a second barrier) folds h_c <- exp(A S) h_c + sum_j w_j x_j B_j^T from
//    the tile in shared memory and stores it.
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

__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kSmallCompute) : "memory");
}
// the first barrier: the compute warps wait, the bookkeeping warp only arrives
__device__ __forceinline__ void meta_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kSmallThreads) : "memory"); }
__device__ __forceinline__ void meta_arrive() {
    asm volatile("bar.arrive 2, %0;" ::"n"(kSmallThreads) : "memory");
}

__global__ void __launch_bounds__(kSmallThreads, 4) m2_decode_small(const M2Args a) {
    constexpr int N = kSmallN, P = kSmallP, VPT = 8, G4 = N / 4, KMX = kMaxL + 1;
    constexpr int CX = P / 8, CB = N / 8;                // 16-byte chunks per x / B row
    extern __shared__ __align__(16) float4 s_h[];        // the checkpoint tile [P][N / 4]
    __shared__ __align__(16) uint16_t s_rB[KMX * N];     // the group's B ring by slot; row L: B_t
    __shared__ __align__(16) uint16_t s_rx[kMaxL * P];   // the head's x ring, by slot
    __shared__ __align__(16) uint16_t s_xt[P];           // the current token's x
    __shared__ __align__(16) float s_w[KMX], s_cbs[KMX], s_dot[P];
    __shared__ __align__(16) float s_wx[KMX * P];        // flush: w_j x_j per row
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
        const int nap = (good && !fold) ? CX + nBC : 0;      // 16-byte chunks to append (+ the dt word)
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
        // Arrive on the sequence's counter as soon as the pointers are in; the result
        // is needed only after the hand-over below, so the round trip overlaps it.
        // Ordering without fences: the arrival depends on the loaded pointer values
        // (it is issued only for good ones), so it leaves after they have returned;
        // the commit depends on the last arrival's result, so it leaves after every
        // CTA of the sequence has arrived, i.e. after every read of the old pointers.
        int prior = -1;
        if (good && lane == 0) prior = atomicAdd(a.arrive + sb, 1);
        if (good) {
            // suffix sums of dt over list positions, newest first (position j < ln is
            // slot (hd + j) mod L, position ln the current token): lane j keeps the sum
            // of the positions after j, lane 0 also that of position 32 (ln = 32)
            auto slot_of = [&](int j) { return hd + j < L ? hd + j : hd + j - L; };
            float acc = 0.0f, sf = 0.0f, sf32 = 0.0f;
#pragma unroll 4
            for (int i = ln; i >= 0; --i) {
                const float di = __shfl_sync(0xffffffffu, rdt, i < ln ? slot_of(i) : 0);
                if (lane == i) sf = acc;
                if (i == 32) sf32 = acc;
                acc += i < ln ? di : dtt;
            }
            // w_j = exp(A S_j) dt_j and exp(A S)
            const int jl = lane < ln ? slot_of(lane) : 0;
            const float dj = __shfl_sync(0xffffffffu, rdt, jl);
            if (lane <= ln) s_w[lane] = expf(Ah * sf) * (lane < ln ? dj : dtt);
            if (lane == 0 && ln == 32) s_w[32] = expf(Ah * sf32) * dtt;
            if (lane == 0) s_dec = expf(Ah * acc);
        }
        if (lane == 0) {
            s_meta[0] = hd;
            s_meta[1] = ln;
        }
        __syncwarp();
        meta_arrive();                                   // pointers, w and exp(A S) are in place
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
    // Three groups of copies, each thread its own share: (0) the float4s of the tile
    // this thread reads below, (1) the B chunks this lane multiplies with C_t below
    // (row r of the group's B ring for every slot r < L, row L the current B_t; 8
    // lanes per row, 16 columns per lane, 4 rows per warp and pass), (2) the x ring
    // and x_t, read by other threads after the barrier.
    const float4 *ck = reinterpret_cast<const float4 *>(a.ckpt) + bh * P * G4;
    for (int v = 0; v < VPT; ++v) {
        const int e = (cw * VPT + v) * G4 + lane;
        cp_async16(s_h + e, ck + e);
    }
    cp_async_commit();
    const int c0 = (lane & 7) * 16;                      // this lane's B / C columns
    const uint16_t *gB = static_cast<const uint16_t *>(a.rec_B) + bg * L * N;
    const uint16_t *gBt = static_cast<const uint16_t *>(a.Bin) + ((size_t)b * G + g) * N;
    for (int rb = 4 * cw; rb <= L; rb += 4 * (kSmallCompute / 32)) {
        const int r = rb + (lane >> 3);
        if (r <= L) {
            const uint16_t *src = (r < L ? gB + r * N : gBt) + c0;
            cp_async16(s_rB + r * N + c0, src);
            cp_async16(s_rB + r * N + c0 + 8, src + 8);
        }
    }
    cp_async_commit();
    {
        const uint16_t *gx = static_cast<const uint16_t *>(a.rec_x) + bh * L * P;
        for (int idx = tid; idx < L * CX + CX; idx += kSmallCompute) {
            if (idx < L * CX) cp_async16(s_rx + idx * 8, gx + idx * 8);
            else cp_async16(s_xt + (idx - L * CX) * 8, static_cast<const uint16_t *>(a.x) + ((size_t)b * H + h) * P +
                                                           (idx - L * CX) * 8);
        }
    }
    cp_async_commit();
    // C_t: this lane's 4 columns of the row dot products, its 16 columns of B . C
    // (through L1: every warp of the CTA reads the same 256 bytes)
    const uint16_t *gC = static_cast<const uint16_t *>(a.Cin) + ((size_t)b * G + g) * N;
    const uint2 craw = __ldg(reinterpret_cast<const uint2 *>(gC) + lane);
    const uint4 q0 = __ldg(reinterpret_cast<const uint4 *>(gC + c0));
    const uint4 q1 = __ldg(reinterpret_cast<const uint4 *>(gC + c0 + 8));
    cp_async_wait_group<1>();                            // this thread's tile values and B chunks
    {
        // h_c . C_t of the warp's rows
        const float4 cfr = make_float4(bf16lo(craw.x), bf16hi(craw.x), bf16lo(craw.y), bf16hi(craw.y));
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
        if (reduced_writer<G4, VPT>()) s_dot[cw * VPT + reduced_index<G4, VPT>(0)] = part[0];
    }
    // B_r . C_t for every ring slot r and B_t (row L), by slot: the ring pointers are
    // not needed yet.  16 columns per lane as bf16 pairs, then a 3-level butterfly.
    for (int rb = 4 * cw; rb <= L; rb += 4 * (kSmallCompute / 32)) {
        const int r = rb + (lane >> 3);
        float acc = 0.0f;
        if (r <= L) {
            const uint4 b0 = *reinterpret_cast<const uint4 *>(s_rB + r * N + c0);
            const uint4 b1 = *reinterpret_cast<const uint4 *>(s_rB + r * N + c0 + 8);
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
        if (r <= L && (lane & 7) == 0) s_cbs[r] = acc;
    }
    cp_async_wait_all();
    meta_sync();                                         // records staged; pointers, w, exp(A S) known
    const int hd = s_meta[0], ln = s_meta[1];
    if (hd < 0 || hd >= L || ln < 0 || ln > L) return;   // flagged by the bookkeeping warp
    const int nrec = ln + 1;
    const bool fold = ln + 1 >= L;
    // list position j < ln is ring slot (hd + j) mod L; j = ln is the current token
    // (row L of the staged B, x_t)
    auto slot_of = [&](int j) { return hd + j < L ? hd + j : hd + j - L; };
    auto brow = [&](int j) { return j < ln ? slot_of(j) : L; };
    auto xrow = [&](int j) -> const uint16_t * { return j < ln ? s_rx + slot_of(j) * P : s_xt; };
    const float dec = s_dec;
    if (tid < P) {
        // the record term of row tid, sum_j w_j (B_j . C_t) x_j + D x_t, then y
        const int row = tid;
        float acc = 0.0f;
#pragma unroll 4
        for (int j = 0; j < nrec; ++j) acc = fmaf(s_w[j] * s_cbs[brow(j)], bf16_at(xrow(j), row), acc);
        const float rt = fmaf(Dh, bf16_at(s_xt, row), acc);
        a.y[((size_t)b * H + h) * P + row] = fmaf(dec, s_dot[row], rt);
    }
    if (!fold) return;

    // flush: w_j x_j for every row, then the rank-nrec update and the decayed
    // checkpoint in one fma per element (the state is rounded once per flush)
    for (int idx = tid; idx < nrec * P; idx += kSmallCompute) {
        const int j = idx / P, row = idx - j * P;
        s_wx[idx] = s_w[j] * bf16_at(xrow(j), row);
    }
    compute_sync();
    // four rows at a time (half the accumulators of the warp's 8 rows live at once)
    const unsigned long long dd = f2pack(dec, dec);
    float4 *cko = reinterpret_cast<float4 *>(a.ckpt) + bh * P * G4;
    for (int r0 = cw * VPT; r0 < cw * VPT + VPT; r0 += 4) {
        unsigned long long acc01[4], acc23[4];           // packed (x, y) and (z, w)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc01[v] = acc23[v] = 0ull;
        for (int j = 0; j < nrec; ++j) {
            const uint2 braw = *reinterpret_cast<const uint2 *>(s_rB + brow(j) * N + lane * 4);
            const unsigned long long b01 = f2pack(bf16lo(braw.x), bf16hi(braw.x));
            const unsigned long long b23 = f2pack(bf16lo(braw.y), bf16hi(braw.y));
            const float4 wa = *reinterpret_cast<const float4 *>(s_wx + j * P + r0);
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
            const int e = (r0 + v) * G4 + lane;
            const float4 hv = s_h[e];
            float4 o;
            f2unpack(fma2(dd, f2pack(hv.x, hv.y), acc01[v]), o.x, o.y);
            f2unpack(fma2(dd, f2pack(hv.z, hv.w), acc23[v]), o.z, o.w);
            __stcg(cko + e, o);
        }
    }
}

}  // namespace

// Batches up to this many sequences take the single-pass kernel: measured (us per
// step, CUDA graphs of 64 steps, this kernel / the persistent kernel) at batch 8
// 8.75 / 12.56, 16 14.97 / 18.17, 32 33.07 / 28.88.
constexpr int kSmallBatchMax = 16;

// Returns RSSM_ERR_UNSUPPORTED (without launching) when the call is not one this
// kernel handles: another shape, a read copy, an FP16 checkpoint, or a batch
// above kSmallBatchMax.
rssm_status launch_decode_small(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st) {
    if (!d->io_bf16 || d->dstate != kSmallN || d->headdim != kSmallP || d->read_copy || d->ckpt_f16)
        return RSSM_ERR_UNSUPPORTED;
    if (d->batch > kSmallBatchMax || d->L > kMaxL) return RSSM_ERR_UNSUPPORTED;
    M2Args a = args;
    void *params[] = {&a};
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
    if (cudaLaunchKernel((const void *)m2_decode_small, dim3(d->nheads, d->batch), dim3(kSmallThreads), params, smem,
                         st) != cudaSuccess)
        return RSSM_ERR_CUDA;
    return launch_status();
}

}  // namespace rssm
