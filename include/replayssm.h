/*
 * replayssm.h -- C ABI of the ReplaySSM decode-state library (libreplayssm.so).
 *
 * The method (three web pages: AT Pulse, "NVIDIA and Princeton's ReplaySSM
 * stores a checkpoint and recent inputs instead of full SSM state to speed up
 * hybrid-model decoding"; The Clarity, "NVIDIA and Princeton cache SSM inputs
 * in place of state to speed hybrid-model decoding"; WittyWires, "ReplaySSM
 * cuts memory traffic to speed up hybrid-model decoding") keeps each
 * sequence's SSM state as a high-precision checkpoint plus a buffer of at most
 * L per-token input records.  Normal decode steps compute the output from the
 * checkpoint and the buffer and write only the new record; every L steps a
 * flush folds the buffer into the checkpoint (AT Pulse §What happened,
 * §Technical analysis "core idea"; Clarity claim ledger [17], [18], [22]).
 * Speculative verify scores draft tokens from the same data and rollback is a
 * buffer-pointer move (AT Pulse §Technical analysis "speculative decoding").
 * A low-precision copy of the checkpoint may serve the reads while the FP32
 * checkpoint drives the recurrence (AT Pulse §Technical analysis
 * "quantization").  The conventional in-place decode, which loads and stores
 * the whole state every step (Clarity claim ledger [6], [7]), and the
 * conventional snapshot-per-draft verify (Clarity claim ledger [13]) are kept
 * as comparison paths.
 *
 * Conventions for every entry point:
 *  - Every pointer is a DEVICE pointer unless said otherwise; every buffer is
 *    allocated and owned by the caller, dense (C order, the layouts below) and
 *    16-byte aligned.  The library allocates nothing and keeps no state.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    stream-ordered and asynchronous: it validates its arguments on the host,
 *    enqueues its kernel (a verify at serving shapes enqueues two), and
 *    returns without synchronising.
 *  - Host-detectable errors (NULL or misaligned pointers, unsupported shapes,
 *    T out of range) return a status before anything is enqueued.  A failed
 *    launch returns RSSM_ERR_CUDA.  Metadata that only the device can see to
 *    be bad (a ring pointer out of range, an accepted count above T) makes the
 *    kernel leave that sequence untouched and OR an RSSM_DEVERR_* bit into
 *    *err.  Kernels never trap; the only thing a kernel ever waits for is its
 *    own asynchronous copies, and those waits give up after ~2 s
 *    (RSSM_DEVERR_TIMEOUT).
 *  - Calls that touch the same cache must be ordered on one stream (the
 *    per-sequence arrival counters below are shared by every call).
 *
 * Mamba-2 notation (per sequence b, head h, group g(h) = h / (nheads/ngroups)):
 *   state h_c[h][p][n] (p < headdim, n < dstate); token inputs dt[h] > 0,
 *   x[h][p], B[g][n], C[g][n]; parameters A[h] < 0, D[h].  One stepwise update
 *   is h <- exp(dt*A) h + dt x B^T, y = h C + D x.  With the checkpoint h_c
 *   taken before records j = 1..k (k = the current token) and S_j the running
 *   sum of dt, the replay output is
 *     y = exp(A S_k) (h_c C) + sum_j exp(A (S_k - S_j)) dt_j (B_j . C) x_j + D x.
 */
#ifndef REPLAYSSM_H
#define REPLAYSSM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RSSM_OK = 0,
    RSSM_ERR_NULL = 1,        /* a required pointer is NULL */
    RSSM_ERR_ALIGN = 2,       /* a pointer is not 16-byte aligned */
    RSSM_ERR_SHAPE = 3,       /* a size is out of the supported range */
    RSSM_ERR_RING = 4,        /* T outside [1, min(L, 8)] */
    RSSM_ERR_CUDA = 5,        /* the kernel launch failed (cudaGetLastError) */
    RSSM_ERR_UNSUPPORTED = 6  /* a supported-but-not-built combination */
} rssm_status;

/* Bits that kernels OR into the caller's *err word. */
#define RSSM_DEVERR_RING_META 0x1u /* ring_head/ring_len out of range: sequence skipped */
#define RSSM_DEVERR_ROLLBACK  0x2u /* accepted outside [0,T] or ring_len < T - accepted */
#define RSSM_DEVERR_SLOT      0x4u /* snapshot slot outside [0, T], or cache slot outside [0, capacity) */
#define RSSM_DEVERR_TIMEOUT   0x8u /* an asynchronous tile copy did not complete within ~2 s;
                                      the kernel abandoned the rest of its work and the
                                      cache (and its arrival counters) must be reset */

/* ------------------------------------------------------------------------ */
/* Mamba-2                                                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t batch;      /* sequences, 1..65535 */
    int32_t nheads;     /* H, multiple of ngroups */
    int32_t headdim;    /* P, multiple of 8, <= 256; headdim * dstate a multiple of 256 */
    int32_t dstate;     /* N, one of 16, 32, 64, 128 */
    int32_t ngroups;    /* G */
    int32_t L;          /* ring capacity = flush threshold, 1..32 */
    int32_t read_copy;  /* 0: reads use the FP32 checkpoint; 1: FP8 E4M3 read copy;
                           2: NVFP4 read copy (E2M1 codes, E4M3 scale per 16 columns) */
    int32_t io_bf16;    /* 1: x, B, C and their records are bf16; 0: float32 */
    int32_t ckpt_f16;   /* 0: FP32 checkpoint; 1: FP16 checkpoint, rounded stochastically
                           at every flush (the random integers come from Philox4x32-10
                           keyed by cache->sr_seed) */
} rssm_mamba2_dims;

typedef struct {
    void     *ckpt;       /* [batch][nheads][headdim][dstate] checkpoint h_c: float32, or
                             FP16 (IEEE binary16) when dims->ckpt_f16 = 1 */
    uint8_t  *ckpt_q;     /* read_copy = 1: [batch][nheads][headdim][dstate] E4M3 codes;
                             read_copy = 2: per (sequence, head) headdim*dstate*9/16 bytes,
                             the E2M1 codes [headdim][dstate/2] (column 2i in the low
                             nibble of byte i) then the E4M3 block scales
                             [headdim][dstate/16] */
    float    *ckpt_scale; /* [batch][nheads][headdim] one float32 scale per row (read_copy 1, 2) */
    float    *rec_dt;     /* [batch][nheads][L] */
    void     *rec_x;      /* [batch][nheads][L][headdim], bf16 or float32 per io_bf16 */
    void     *rec_B;      /* [batch][ngroups][L][dstate] */
    void     *rec_C;      /* [batch][ngroups][L][dstate]; NULL = C is not kept */
    int32_t  *ring_head;  /* [batch] ring slot of the oldest buffered record, [0, L) */
    int32_t  *ring_len;   /* [batch] buffered records, [0, L] */
    int32_t  *arrive;     /* [batch] scratch counters: zero before the first call,
                             every call leaves them zero again */
    const float *A;       /* [nheads] */
    const float *D;       /* [nheads] */
    uint32_t *err;        /* one word; RSSM_DEVERR_* bits are ORed in */
    /* Cache-slot indirection (engine-style state indices; continuous batching):
     * the cache arrays above hold `capacity` sequences ([capacity] in place of
     * [batch] in their layouts) and batch row b of a call's inputs and outputs
     * belongs to the sequence in slot slots[b].  slots == NULL: row b uses slot b.
     * capacity == 0: capacity = batch.  The slots of one call must be distinct.
     * A slot outside [0, capacity) skips that row and sets RSSM_DEVERR_SLOT. */
    const int32_t *slots; /* [batch] device, or NULL */
    int32_t capacity;
    /* Seed of this call's stochastic rounding (dims->ckpt_f16 = 1): the element
     * in column n, row p of head h of cache slot s takes 16 random bits from
     * Philox4x32-10 with counter (n/8, p, h, s) and key (seed mod 2^32,
     * seed / 2^32), half n mod 2 of output word (n mod 8)/2.  Pass a new seed
     * to every call that may flush (decode, verify, flush), e.g. a step count:
     * a repeated seed repeats the rounding decisions. */
    uint64_t sr_seed;
} rssm_mamba2_cache;

/*
 * Replay decode of one token per sequence (AT Pulse §What happened: normal
 * steps compute each output from the checkpoint plus the buffered records and
 * write only the new record; Clarity claim ledger [18]).
 *   dt [batch][nheads] f32; x [batch][nheads][headdim]; B, C
 *   [batch][ngroups][dstate] (bf16 or f32 per io_bf16); y [batch][nheads][headdim] f32.
 * With len = ring_len[b] records buffered:
 *   len + 1 <  L: append (dt, x, B, C) at slot (ring_head + len) mod L,
 *                 ring_len += 1; the checkpoint is only read.
 *   len + 1 >= L: flush fused into this step (AT Pulse §Technical analysis:
 *                 every L steps the buffer is folded into the checkpoint):
 *                 h_c <- exp(A S) h_c + sum_j exp(A (S - S_j)) dt_j x_j B_j^T
 *                 over the buffered records and the current token (computed in
 *                 float32; an FP16 checkpoint is then rounded stochastically with
 *                 cache->sr_seed), the read copy is re-quantised from the stored
 *                 checkpoint, ring_head <- (ring_head + len + 1) mod L,
 *                 ring_len <- 0; the current token is not stored.
 * y is the replay output above in every case.  Non-flush steps read the FP8
 * copy when dims->read_copy = 1 and the NVFP4 copy when it is 2.
 */
rssm_status replayssm_decode(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                             const float *dt, const void *x, const void *B, const void *C,
                             float *y, void *stream);

/*
 * replayssm_decode for callers that cannot allocate device memory (the paper
 * has no counterpart; this is a library convenience).  Some callers cannot
 * call cudaMalloc or keep a buffer of their own between calls -- for example
 * a plugin inside an inference engine whose memory planner owns all device
 * memory and passes the plugin only its inputs and outputs -- so they have no
 * place for the per-sequence arrival counters that replayssm_decode takes in
 * cache->arrive.  This entry point ignores cache->arrive (it may be NULL) and
 * uses a fixed array of 4096 counters (16 KiB) in the library's own device
 * memory instead; every GPU that loads the library holds that array until
 * the process exits.  Everything else -- arguments, results, errors -- is as
 * replayssm_decode.
 *  - batch (or, with a slot map, the cache capacity) > 4096 returns RSSM_ERR_SHAPE
 *    before anything is enqueued.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - The first call on a device looks up the array's device address with that
 *    device current; make that first call before any stream capture.  The
 *    address is kept until the process exits, so do not use this entry point
 *    after a cudaDeviceReset (or any other teardown of the device's primary
 *    context) in the same process.
 *  - Every host-side check of replayssm_decode runs before anything is
 *    enqueued, so a rejected call leaves the shared counters untouched.
 *  - Each call clears the counters it uses (an asynchronous memset on
 *    `stream`) and then enqueues the decode.
 *  - All calls share the one array: calls that can overlap on the GPU (other
 *    streams, other host threads) race on it and must be serialised.
 */
rssm_status replayssm_decode_noalloc(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                                     const float *dt, const void *x, const void *B, const void *C,
                                     float *y, void *stream);

/*
 * Test hook of the failure-detection path (the pages have no counterpart):
 * replayssm_decode at a serving shape (persistent kernel, FP32 checkpoint),
 * except that the consumer warps first wait on a barrier that nothing arrives
 * on.  That wait gives up after ~2 s like every wait in the kernels, so the
 * kernel takes its abort path on a healthy GPU: it sets RSSM_DEVERR_TIMEOUT in
 * *cache->err, lets every copy it started land, and exits.  The ring pointers
 * are committed at kernel start as usual, but outputs, records and the
 * checkpoint are left partly written: the cache is not usable afterwards.
 * Arguments and host-side errors are those of replayssm_decode;
 * RSSM_ERR_UNSUPPORTED for shapes the persistent kernel does not serve.
 */
rssm_status replayssm_test_stalled_decode(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                                          const float *dt, const void *x, const void *B, const void *C,
                                          float *y, void *stream);

/*
 * Standalone flush (WittyWires §What happened: the checkpoint is updated when
 * the buffer fills): for every sequence with mask[b] != 0 (mask = NULL: all),
 * fold its ring_len records into the checkpoint with the same arithmetic as
 * the fused flush (FP16 checkpoints rounded stochastically with cache->sr_seed),
 * re-quantise the read copy, ring_head <- (ring_head + ring_len) mod L,
 * ring_len <- 0.  mask is a device array of batch bytes.
 */
rssm_status replayssm_flush(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                            const uint8_t *mask, void *stream);

/*
 * Speculative verify of T drafts per sequence by output-only evaluation
 * (AT Pulse §Technical analysis "speculative decoding": no intermediate state
 * is built).  dt [batch][T][nheads]; x [batch][T][nheads][headdim]; B, C
 * [batch][T][ngroups][dstate]; y [batch][T][nheads][headdim] f32.
 * If ring_len + T > L the buffered records are folded first (as
 * replayssm_flush).  Draft i (1-based) is scored against the checkpoint, the
 * buffered records and drafts 1..i; the T drafts are appended at slots
 * (ring_head + ring_len + i - 1) mod L and ring_len += T.  Drafts are never
 * folded by a verify.  1 <= T <= min(L, 8).  Reads use the checkpoint itself
 * (float32 or FP16), not the read copy.
 */
rssm_status replayssm_verify(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                             int32_t T, const float *dt, const void *x, const void *B,
                             const void *C, float *y, void *stream);

/*
 * Rollback after a verify of T drafts (AT Pulse §Technical analysis: rolling
 * back rejected drafts is a buffer-pointer move): ring_len[b] -= T -
 * accepted[b].  accepted [batch] int32 in [0, T]; a sequence with an accepted
 * count outside that range, or fewer than T - accepted records, is left as it
 * is and RSSM_DEVERR_ROLLBACK is raised.  No state or record bytes move.
 */
rssm_status replayssm_rollback(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                               int32_t T, const int32_t *accepted, void *stream);

/*
 * (Re)build the read copy from the FP32 checkpoint for every sequence (AT
 * Pulse §Technical analysis "quantization": a high-precision checkpoint drives
 * the recurrence, a low-precision copy serves the reads).
 * FP8 (read_copy 0 or 1): per (head, row) amax = max|h|, scale = amax/448,
 * code = E4M3 round-to-nearest-even, saturating, of h * (448/amax); a zero row
 * gets scale 1 and zero codes.
 * NVFP4 (read_copy 2; AT Pulse §What happened: 4-bit NVFP4 reads; the block
 * layout is the format's public definition): per row s_r = amax/2688 and
 * k_r = 448/amax; per 16-column block with maximum m, block scale code
 * E4M3(m * k_r), d = e4m3(code) * s_r, element code E2M1 round-to-nearest-
 * even, saturating, of h * (1/d); every step one correctly rounded float32
 * operation; a zero row stores zero codes, zero block scales and s_r = 0.
 * Used once after the checkpoint is initialised; flushes keep the copy
 * current afterwards.
 */
rssm_status replayssm_requant(const rssm_mamba2_dims *dims, const rssm_mamba2_cache *cache,
                              void *stream);

/*
 * Conventional in-place decode (Clarity claim ledger [6]: each step updates
 * the state, reads the output from it and stores it): state
 * [batch][nheads][headdim][dstate] f32 is loaded, updated
 * h <- exp(dt A) h + dt x B^T, contracted y = h C + D x, and stored back.
 * Inputs as replayssm_decode.  dims->L and read_copy are ignored.
 */
rssm_status replayssm_conventional_decode(const rssm_mamba2_dims *dims, float *state,
                                          const float *A, const float *D, const float *dt,
                                          const void *x, const void *B, const void *C,
                                          float *y, void *stream);

/*
 * Conventional speculative verify with a snapshot per draft (Clarity claim
 * ledger [13]: one state read and T state writes per step).  pool is
 * [batch][T+1][nheads][headdim][dstate] f32; slot [batch] int32 names the
 * pool entry holding the current state.  The T drafts are applied stepwise;
 * the state after draft i is stored in entry (slot + i) mod (T + 1) and y of
 * draft i is read from it.  Inputs/outputs as replayssm_verify.  A slot
 * outside [0, T] raises RSSM_DEVERR_SLOT and the sequence is skipped.
 */
rssm_status replayssm_conventional_verify(const rssm_mamba2_dims *dims, float *pool,
                                          const int32_t *slot, int32_t T, const float *A,
                                          const float *D, const float *dt, const void *x,
                                          const void *B, const void *C, float *y,
                                          uint32_t *err, void *stream);

/*
 * Conventional rollback: slot[b] <- (slot[b] + accepted[b]) mod (T + 1), i.e.
 * keep the snapshot after the accepted prefix (0 = the state before the
 * drafts).  An accepted count outside [0, T] raises RSSM_DEVERR_ROLLBACK.
 */
rssm_status replayssm_conventional_select(int32_t batch, int32_t *slot, int32_t T,
                                          const int32_t *accepted, uint32_t *err, void *stream);

/* ------------------------------------------------------------------------ */
/* Gated DeltaNet (gated delta rule)                                          */
/* ------------------------------------------------------------------------ */
/*
 * Per sequence and head: state S[dv][dk]; token (q, k in R^dk, v in R^dv,
 * alpha, beta scalars):  S <- alpha S (I - beta k k^T) + beta v k^T,  o = S q
 * (AT Pulse §Capabilities and access: Gated DeltaNet kernels; the replay idea
 * of §Technical analysis applied to the gated delta rule).  Replay form with
 * checkpoint S_c and records j = 1..k (k = current): u_k = q,
 * u_{j-1} = alpha_j (u_j - beta_j k_j (k_j . u_j)),
 * o = S_c u_0 + sum_j beta_j (k_j . u_j) v_j.
 */
typedef struct {
    int32_t batch;
    int32_t nheads;
    int32_t dk;    /* one of 16, 32, 64, 128 */
    int32_t dv;    /* multiple of 8, <= 256; dk * dv a multiple of 256 */
    int32_t L;     /* 1..32 */
} rssm_gdn_dims;

typedef struct {
    float    *ckpt;       /* [batch][nheads][dv][dk] FP32 checkpoint S_c */
    uint16_t *rec_k;      /* [batch][nheads][L][dk] bf16 */
    uint16_t *rec_v;      /* [batch][nheads][L][dv] bf16 */
    float    *rec_alpha;  /* [batch][nheads][L] */
    float    *rec_beta;   /* [batch][nheads][L] */
    int32_t  *ring_head;  /* [batch] */
    int32_t  *ring_len;   /* [batch] */
    int32_t  *arrive;     /* [batch] scratch counters, zero before the first call */
    uint32_t *err;
    /* Cache-slot indirection, as for the Mamba-2 cache: the arrays above hold
     * `capacity` sequences and batch row b uses slot slots[b] (NULL: slot b;
     * capacity 0: batch; distinct slots per call; an out-of-range slot skips
     * its row and sets RSSM_DEVERR_SLOT). */
    const int32_t *slots; /* [batch] device, or NULL */
    int32_t capacity;
} rssm_gdn_cache;

/*
 * GDN replay decode, same ring rules as replayssm_decode (fused flush when
 * ring_len + 1 >= L folds the records and the current token row by row:
 * s <- alpha_j (s - beta_j (s . k_j) k_j) + beta_j v_j[r] k_j).
 * q, k [batch][nheads][dk] bf16; v [batch][nheads][dv] bf16; alpha, beta
 * [batch][nheads] f32; o [batch][nheads][dv] f32.
 */
rssm_status replayssm_gdn_decode(const rssm_gdn_dims *dims, const rssm_gdn_cache *cache,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *alpha, const float *beta, float *o, void *stream);

/* GDN standalone flush of the masked sequences (mask NULL = all). */
rssm_status replayssm_gdn_flush(const rssm_gdn_dims *dims, const rssm_gdn_cache *cache,
                                const uint8_t *mask, void *stream);

/*
 * GDN speculative verify (AT Pulse, Technical analysis: the drafts are scored by
 * output-only evaluation from the checkpoint and the buffered inputs; Capabilities
 * and access: the method's kernels cover speculative decoding): draft i of each
 * sequence is scored causally from the checkpoint, the buffered records and drafts
 * 1..i, i.e. o_i = S_c u_0 + sum_j beta_j (k_j . u_j) v_j with the backward chain
 * started from q_i at draft i.  Nothing is folded on account of the drafts; when
 * ring_len + T > L the buffered records are first folded into the checkpoint (the
 * pre-flush) so that the T drafts fit.  The drafts' records are appended and
 * ring_len grows by T (a second, small kernel writes them after the first, because
 * on a pre-flush they land on slots the first still reads).
 * T in 1..8 and T <= L; q, k [batch][T][nheads][dk] bf16; v [batch][T][nheads][dv]
 * bf16; alpha, beta [batch][T][nheads] f32; o [batch][T][nheads][dv] f32.
 * Errors: RSSM_ERR_RING for T out of range, otherwise as replayssm_gdn_decode.
 */
rssm_status replayssm_gdn_verify(const rssm_gdn_dims *dims, const rssm_gdn_cache *cache, int32_t T,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *alpha, const float *beta, float *o, void *stream);

/*
 * GDN rollback after a verify of T drafts (AT Pulse, Technical analysis: rollback is
 * a buffer-pointer move): ring_len[b] -= T - accepted[b], accepted [batch] int32 in
 * 0..T on the device.  A sequence whose accepted count is out of range, or whose ring
 * holds fewer than T - accepted records, is left as it is and RSSM_DEVERR_ROLLBACK is
 * set in the error word.
 */
rssm_status replayssm_gdn_rollback(const rssm_gdn_dims *dims, const rssm_gdn_cache *cache, int32_t T,
                                   const int32_t *accepted, void *stream);

/* GDN conventional in-place decode of state [batch][nheads][dv][dk] f32. */
rssm_status replayssm_gdn_conventional_decode(const rssm_gdn_dims *dims, float *state,
                                              const uint16_t *q, const uint16_t *k,
                                              const uint16_t *v, const float *alpha,
                                              const float *beta, float *o, void *stream);

/* ------------------------------------------------------------------------ */

/* Static string for a status code (host). */
const char *replayssm_status_string(rssm_status s);

/* Library ABI version: 0x00MMmmpp. */
uint32_t replayssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* REPLAYSSM_H */
