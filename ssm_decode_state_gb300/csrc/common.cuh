// Device helpers shared by the ReplaySSM kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "replayssm.h"

namespace rssm {

constexpr int kMaxL = 32;   // ring capacity limit
constexpr int kMaxT = 8;    // drafts per verify limit

// ---------------------------------------------------------------- loads/stores

// Streaming (evict-first) 16-byte load/store for checkpoint tiles: each tile
// is touched once per step, so it should not push the ring records out of L2.
__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }
__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t *p) { return __ldcs(p); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// A 16-byte chunk of an input or record row holds 8 bf16 or 4 float32 values.
__device__ __forceinline__ void unpack_chunk(uint4 c, bool bf16, float *out) {
    if (bf16) {
        out[0] = bf16lo(c.x); out[1] = bf16hi(c.x);
        out[2] = bf16lo(c.y); out[3] = bf16hi(c.y);
        out[4] = bf16lo(c.z); out[5] = bf16hi(c.z);
        out[6] = bf16lo(c.w); out[7] = bf16hi(c.w);
    } else {
        out[0] = __uint_as_float(c.x); out[1] = __uint_as_float(c.y);
        out[2] = __uint_as_float(c.z); out[3] = __uint_as_float(c.w);
    }
}

// --------------------------------------------------------------- reductions

// Sum V per-lane values over aligned groups of G lanes (G, V powers of two,
// G <= 32) with V/2 + V/4 + ... shuffles instead of V*log2(G): each round
// every lane keeps one half of its values and trades the other half with its
// partner.  On return:
//   V <= G: v[0] holds the group sum of value index (lane % G) / (G / V);
//   V >  G: v[i] (i < V/G) holds the group sum of value (lane % G) * (V/G) + i.
template <int O, int C, int V, bool kMax = false>
struct GroupReduce {
    static __device__ __forceinline__ float op(float a, float b) { return kMax ? fmaxf(a, b) : a + b; }
    static __device__ __forceinline__ void run(float (&v)[V], int lane) {
        if constexpr (O >= 1) {
            if constexpr (C > 1) {
                const bool up = (lane & O) != 0;
#pragma unroll
                for (int i = 0; i < C / 2; ++i) {
                    const float send = up ? v[i] : v[i + C / 2];
                    const float keep = up ? v[i + C / 2] : v[i];
                    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, O));
                }
                GroupReduce<O / 2, C / 2, V, kMax>::run(v, lane);
            } else {
                v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], O));
                GroupReduce<O / 2, 1, V, kMax>::run(v, lane);
            }
        }
    }
};

template <int G, int V>
__device__ __forceinline__ void group_reduce(float (&v)[V]) {
    GroupReduce<G / 2, V, V>::run(v, threadIdx.x & 31);
}

// The same exchange pattern with max instead of sum (same result placement).
template <int G, int V>
__device__ __forceinline__ void group_reduce_max(float (&v)[V]) {
    GroupReduce<G / 2, V, V, true>::run(v, threadIdx.x & 31);
}

// Value index of v[i] after group_reduce<G, V>, and whether this lane is the
// one (of the G/V lanes holding the same sum) that should publish it.
template <int G, int V>
__device__ __forceinline__ int reduced_index(int i) {
    const int lg = threadIdx.x & (G - 1);
    if constexpr (V <= G) return lg / (G / V);
    else return lg * (V / G) + i;
}
template <int G, int V>
__device__ __forceinline__ bool reduced_writer() {
    if constexpr (V <= G) return (threadIdx.x & (G / V - 1)) == 0;
    else return true;
}

// Like group_reduce, but every lane of the group ends with all V sums in v.
template <int G, int V>
__device__ __forceinline__ void group_allreduce(float (&v)[V]) {
    float t[V];
#pragma unroll
    for (int i = 0; i < V; ++i) t[i] = v[i];
    group_reduce<G, V>(t);
    const int base = (threadIdx.x & 31) & ~(G - 1);
#pragma unroll
    for (int vi = 0; vi < V; ++vi) {
        if constexpr (V <= G) v[vi] = __shfl_sync(0xffffffffu, t[0], base + vi * (G / V));
        else v[vi] = __shfl_sync(0xffffffffu, t[vi % (V / G)], base + vi / (V / G));
    }
}

template <int G>
__device__ __forceinline__ float group_max(float x) {
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// ----------------------------------------------------------------------- FP8

// Four float32 values -> four E4M3 codes (round to nearest even, saturating),
// byte i of the result = element i.
__device__ __forceinline__ uint32_t e4m3_pack4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xffffu) | (hi << 16);
}

// Four E4M3 codes (byte i = element i) -> float4.
__device__ __forceinline__ float4 e4m3_unpack4(uint32_t w) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Four E4M3 codes (byte i = column i) as two pairs of bfloat16 values, even
// columns (0, 2) and odd columns (1, 3), each 2^-120 times the code's value:
// the code's exponent and mantissa bits become the low exponent bits and the
// top mantissa bits of a bfloat16 (normal codes read as normal bfloat16 with
// the bias 120 too large, subnormal codes as bfloat16 subnormals with the same
// offset), integer operations only.  Never given NaN codes (the encoder
// saturates to the largest finite value).
__device__ __forceinline__ void e4m3_to_bf16_pairs(uint32_t w, uint32_t &even, uint32_t &odd) {
    even = ((w & 0x007f007fu) << 4) | ((w << 8) & 0x80008000u);
    odd = ((w & 0x7f007f00u) >> 4) | (w & 0x80008000u);
}

// acc + a.lo * c.lo + a.hi * c.hi: bfloat16 pairs, products exact, FP32
// accumulation (mixed-precision fma of sm_100 and later).
__device__ __forceinline__ float fma_bf16_pair(uint32_t a, uint32_t c, float acc) {
    asm("{ .reg .b16 al, ah, cl, ch;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {cl, ch}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, cl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ah, ch, %0; }"
        : "+f"(acc)
        : "r"(a), "r"(c));
    return acc;
}

// Per-row read-copy scale: scale = amax/448 and inv = 448/amax, each one
// correctly rounded float32 division; a zero row (or one whose inverse
// overflows) is stored as zero codes with scale 1.
__device__ __forceinline__ void e4m3_row_scale(float amax, float &scale, float &inv) {
    inv = __fdiv_rn(448.0f, amax);
    scale = __fdiv_rn(amax, 448.0f);
    if (!(amax > 0.0f) || isinf(inv)) {
        inv = 0.0f;
        scale = 1.0f;
    }
}

// Read-copy codes of V rows held by one warp, 32 lanes per row (lane i holds
// columns 4i..4i+3 of every row).  The row maxima go through one transposed
// exchange, each lane derives scale and inverse for the row it ends up with
// (row (lane / (32/V))), and the inverses are broadcast back: two divisions
// per lane instead of two per row per lane.  Codes and scales are the same
// as per-row e4m3_row_scale + e4m3_pack4.  On return q[v] holds this lane's
// four codes of row v and row_scale the scale of row (lane / (32/V)).
template <int V>
__device__ __forceinline__ void e4m3_quantize_rows(const float4 (&o)[V], uint32_t (&q)[V], float &row_scale) {
    static_assert(V <= 32 && (V & (V - 1)) == 0, "rows per warp");
    float m[V];
#pragma unroll
    for (int v = 0; v < V; ++v) m[v] = fmaxf(fmaxf(fabsf(o[v].x), fabsf(o[v].y)), fmaxf(fabsf(o[v].z), fabsf(o[v].w)));
    group_reduce_max<32, V>(m);
    float inv;
    e4m3_row_scale(m[0], row_scale, inv);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const float iv = __shfl_sync(0xffffffffu, inv, v * (32 / V));
        q[v] = e4m3_pack4(__fmul_rn(o[v].x, iv), __fmul_rn(o[v].y, iv), __fmul_rn(o[v].z, iv), __fmul_rn(o[v].w, iv));
    }
}

// --------------------------------------------------------------------- NVFP4
//
// NVFP4 read copy: E2M1 element codes (OCP Microscaling Formats: 1 sign bit,
// 2 exponent bits with bias 1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2,
// 3, 4, 6), one E4M3 scale per 16 consecutive columns of a row and one float32
// scale per row.  One head's copy is its codes [P][N/2] (column 2i in the low
// nibble of byte i) followed by its block scales [P][N/16].

constexpr float kNv4RowTarget = 2688.0f;    // 6 (largest E2M1) x 448 (largest E4M3)

__host__ __device__ constexpr int nv4_head_bytes(int P, int N) { return P * N / 2 + P * N / 16; }

// Row scale s_r = amax / 2688 and the block-scale factor k_r = 448 / amax,
// each one correctly rounded float32 division; a zero row, or one whose
// scales leave the float32 range, gets s_r = k_r = 0 (every block scale 0).
__device__ __forceinline__ void nv4_row_scale(float amax, float &s_r, float &k_r) {
    s_r = __fdiv_rn(amax, kNv4RowTarget);
    k_r = __fdiv_rn(448.0f, amax);
    if (!(amax > 0.0f) || !(s_r > 0.0f) || isinf(k_r)) {
        s_r = 0.0f;
        k_r = 0.0f;
    }
}

// Value of an E4M3 code as float32, exactly: its exponent and mantissa bits
// placed as the low exponent bits and top mantissa bits of a float32 read
// 2^-120 times the value (subnormal codes as float32 subnormals), then scaled
// back.  Never given NaN codes.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    return __uint_as_float(((code & 0x7fu) << 20) | ((code & 0x80u) << 24)) * 0x1p120f;
}

// Block scale code of a block with largest magnitude amax_c, and the inverse
// of its effective scale e4m3(code) * s_r (0 when that is 0 or its inverse
// overflows).
__device__ __forceinline__ uint32_t nv4_block_scale(float amax_c, float s_r, float k_r, float &inv) {
    const uint32_t code = __nv_cvt_float_to_fp8(__fmul_rn(amax_c, k_r), __NV_SATFINITE, __NV_E4M3);
    const float d = __fmul_rn(e4m3_value(code), s_r);
    inv = d > 0.0f ? __frcp_rn(d) : 0.0f;
    if (isinf(inv)) inv = 0.0f;
    return code;
}

// Four float32 values -> four E2M1 codes (round to nearest even, saturating),
// nibble i of the 16-bit result = element i.
__device__ __forceinline__ uint32_t e2m1_pack4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
    const uint32_t hi = __nv_cvt_float2_to_fp4x2(make_float2(c, d), __NV_E2M1, cudaRoundNearest);
    return (lo & 0xffu) | ((hi & 0xffu) << 8);
}

// Four E2M1 codes (nibble i = element i) -> float4 of their values.  The
// code's exponent and mantissa bits become the low exponent bits and top
// mantissa bit of a float32 that reads 2^-126 times the value (the 0.5 code
// as a float32 subnormal), scaled back exactly.
__device__ __forceinline__ float4 e2m1_unpack4(uint32_t w) {
    float r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t n = (w >> (4 * i)) & 0xfu;
        r[i] = __uint_as_float(((n & 7u) << 22) | ((n & 8u) << 28)) * 0x1p126f;
    }
    return make_float4(r[0], r[1], r[2], r[3]);
}

// Eight E2M1 codes (nibble k = column k) -> their values as four f16 pairs,
// pair i = columns (2i, 2i + 1), by the hardware conversion (E2M1 values are
// exact in f16).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// Four E4M3 codes (byte k = column k) -> their values as two f16 pairs, columns
// (0, 1) and (2, 3), by the hardware conversion (E4M3 values are exact in f16).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const __half2_raw a = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
    const __half2_raw c = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    lo = (uint32_t)a.x | ((uint32_t)a.y << 16);
    hi = (uint32_t)c.x | ((uint32_t)c.y << 16);
}

// D += A B for one 16 x 8 x 16 tile: the warp-level MMA, f16 operands, FP32
// accumulation.  Fragment registers as the PTX ISA lays them out for
// m16n8k16 (A row-major: a0 rows g, a1 rows g + 8, a2 / a3 the same rows at
// k + 8; B column-major: b0 k = 2t, 2t + 1, b1 k + 8; D d0, d1 row g, d2, d3
// row g + 8, columns 2t, 2t + 1; g = lane / 4, t = lane % 4).
__device__ __forceinline__ void mma_f16_16x8x16(float &d0, float &d1, float &d2, float &d3, uint32_t a0,
                                                uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A B for one 16 x 8 x 32 tile of E4M3 operands: the warp-level MMA, FP32
// accumulation.  Each register holds 4 consecutive k of one row of A or one
// column of B: a0 rows g, a1 rows g + 8, k = 4t .. 4t + 3; a2 / a3 the same rows
// at k + 16; b0 column g, k = 4t .. 4t + 3, b1 k + 16; D as for m16n8k16 (g =
// lane / 4, t = lane % 4).  Products of E4M3 values are exact in FP32.
__device__ __forceinline__ void mma_e4m3_16x8x32(float &d0, float &d1, float &d2, float &d3, uint32_t a0,
                                                 uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four floats -> four E4M3 codes (byte k = value k), round to nearest even,
// saturating to the largest finite code, by the hardware conversion.
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float v0, float v1, float v2, float v3) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v2, v3), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// acc + a.lo * c.lo + a.hi * c.hi: f16 pairs, products exact, FP32
// accumulation (mixed-precision fma of sm_100 and later).
__device__ __forceinline__ float fma_f16_pair(uint32_t a, uint32_t c, float acc) {
    asm("{ .reg .b16 al, ah, cl, ch;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {cl, ch}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, cl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, ch, %0; }"
        : "+f"(acc)
        : "r"(a), "r"(c));
    return acc;
}

// 2^e as a float32 for -126 <= e <= 127.
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// NVFP4 copy of 8 rows held by one warp, 32 lanes per row (lane i holds
// columns 4i..4i+3, so the 16-column block c spans lanes 4c..4c+3), written
// to the head's copy hq (codes, then block scales) and row scales rs.  The
// per-(row, block) scalar work is split over the block's 4 lanes: a transposed
// max exchange leaves lane 4c + j with the block maxima of rows 2j and 2j + 1,
// three butterflies across the blocks give those rows' maxima, the lane
// derives both rows' scales and stores their block-scale codes, and the
// inverses go back to the block's lanes by shuffles.  Same float32 operations
// per row and block as nv4_row_scale + nv4_block_scale + e2m1_pack4.
// row_of(v) is the head row of this warp's v-th row.
template <class RowFn>
__device__ __forceinline__ void nv4_quantize_store(const float4 (&o)[8], uint8_t *hq, float *rs, int P, int N,
                                                   RowFn row_of) {
    const int lane = threadIdx.x & 31, c = lane >> 2, j = lane & 3;
    float m[8];
#pragma unroll
    for (int v = 0; v < 8; ++v)
        m[v] = fmaxf(fmaxf(fabsf(o[v].x), fabsf(o[v].y)), fmaxf(fabsf(o[v].z), fabsf(o[v].w)));
    group_reduce_max<4, 8>(m);                           // m[i]: block maximum of row 2j + i
    float r0 = m[0], r1 = m[1];
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        r0 = fmaxf(r0, __shfl_xor_sync(0xffffffffu, r0, x));
        r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, x));
    }
    float s0, k0, s1, k1, inv0, inv1;
    nv4_row_scale(r0, s0, k0);
    nv4_row_scale(r1, s1, k1);
    const uint32_t sb0 = nv4_block_scale(m[0], s0, k0, inv0);
    const uint32_t sb1 = nv4_block_scale(m[1], s1, k1, inv1);
    const int ra = row_of(2 * j), rb = row_of(2 * j + 1);
    hq[P * N / 2 + ra * (N / 16) + c] = (uint8_t)sb0;
    hq[P * N / 2 + rb * (N / 16) + c] = (uint8_t)sb1;
    if (c == 0) {
        rs[ra] = s0;
        rs[rb] = s1;
    }
    const int base = lane & ~3;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const float inv = __shfl_sync(0xffffffffu, (v & 1) ? inv1 : inv0, base + (v >> 1));
        reinterpret_cast<uint16_t *>(hq + row_of(v) * (N / 2))[lane] = (uint16_t)e2m1_pack4(
            __fmul_rn(o[v].x, inv), __fmul_rn(o[v].y, inv), __fmul_rn(o[v].z, inv), __fmul_rn(o[v].w, inv));
    }
}

// ------------------------------------------------------ FP16 checkpoint (SR)
//
// An FP16 checkpoint is rounded stochastically at every flush.  Random
// integers come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC'11): counter (column / 8, row,
// head, cache slot), key = the call's 64-bit seed; the element in column
// 8q + k takes the 16-bit half k mod 2 of output word k / 2.

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// Stochastic rounding of v to FP16 with a 16-bit random integer r: lo = the
// FP16 value at or below |v|, u = the FP16 step above lo, round up when
// r < 65536 (|v| - lo) / u; |v| >= 65504 saturates.  In the normal FP16 range
// (a) (|v| - lo) / u is the 13 float32 mantissa bits below the FP16 mantissa
// over 2^13, so the test is (r >> 3) < those bits and rounding up adds one
// FP16 step to the truncated bit pattern; below it (b) the step is 2^-24 and
// every operation is exact in float32.
__device__ __forceinline__ uint32_t sr_f16(float v, uint32_t r) {
    const uint32_t ub = __float_as_uint(v), sgn = (ub >> 16) & 0x8000u, ab = ub & 0x7fffffffu;
    if (ab >= 0x477fe000u) return sgn | 0x7bffu;                  // |v| >= 65504
    if (ab >= 0x38800000u) {                                      // (a) |v| >= 2^-14
        const uint32_t t = (ab & ~0x1fffu) + ((r >> 3) < (ab & 0x1fffu) ? 0x2000u : 0u);
        return sgn | __half_as_ushort(__float2half_rn(__uint_as_float(t)));
    }
    const float a = __uint_as_float(ab);                          // (b) FP16 subnormals: step 2^-24
    const float lo = __half2float(__float2half_rz(a));
    const float res = __uint2float_rn(r) < (a - lo) * 0x1p40f ? lo + 0x1p-24f : lo;
    return sgn | __half_as_ushort(__float2half_rn(res));
}

// Four consecutive columns rounded stochastically to FP16 with the random
// words w0 (columns 0, 1) and w1 (columns 2, 3), packed low column first; `o`
// becomes the rounded values.
__device__ __forceinline__ uint2 sr_f16x4_words(float4 &o, uint32_t w0, uint32_t w1) {
    const uint32_t e0 = sr_f16(o.x, w0 & 0xffffu), e1 = sr_f16(o.y, w0 >> 16);
    const uint32_t e2 = sr_f16(o.z, w1 & 0xffffu), e3 = sr_f16(o.w, w1 >> 16);
    o = make_float4(__half2float(__ushort_as_half((unsigned short)e0)), __half2float(__ushort_as_half((unsigned short)e1)),
                    __half2float(__ushort_as_half((unsigned short)e2)), __half2float(__ushort_as_half((unsigned short)e3)));
    return make_uint2(e0 | (e1 << 16), e2 | (e3 << 16));
}

// Columns 4c..4c+3 of row `row` of head `head` of cache slot `slot`: one
// generator call for the column group c / 2, words 2 (c mod 2) and 2 (c mod 2) + 1.
__device__ __forceinline__ uint2 sr_f16x4(float4 &o, uint32_t c, uint32_t row, uint32_t head, uint32_t slot,
                                          uint32_t seed_lo, uint32_t seed_hi) {
    const uint4 r = philox4x32_10(make_uint4(c >> 1, row, head, slot), seed_lo, seed_hi);
    return (c & 1) ? sr_f16x4_words(o, r.z, r.w) : sr_f16x4_words(o, r.x, r.y);
}

// Four FP16 values (packed low first) -> float4.
__device__ __forceinline__ float4 f16x4_to_float4(uint2 w) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// ------------------------------------------------------------------ the ring

// Sum of dt[j+1 .. e] accumulated from the newest record backwards (j = -1:
// the whole prefix 0..e).  Every path that needs a decay exponent uses this
// one order, so fused and standalone flushes agree bit for bit.
__device__ __forceinline__ float suffix_sum(const float *dt, int j, int e) {
    float s = 0.0f;
#pragma unroll 4
    for (int m = e; m > j; --m) s += dt[m];
    return s;
}

__device__ __forceinline__ void flag_error(uint32_t *err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

// ------------------------------------------------- async copies (sm_90+ PTX)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// `count` arrivals at once (release semantics, like mbar_arrive).
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// One-dimensional bulk copy global -> this CTA's shared memory (TMA engine);
// completion is signalled on `bar` as transaction bytes.  dst, src and bytes
// must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// The same copy with the default L2 policy (for data that is read again soon).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier, giving up after ~2 s (returns
// false); a copy that never lands must not hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    uint64_t t0 = 0;                                   // the clock is read only in long waits
    for (uint32_t it = 1; it <= (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > 2000000000ull) return false;
        }
    }
    return false;
}

// Ampere-style asynchronous 16- and 4-byte copies into shared memory, for
// small scattered record rows.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Wait until at most NPEND of this thread's committed cp.async groups are pending.
template <int NPEND>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(NPEND) : "memory"); }

}  // namespace rssm
