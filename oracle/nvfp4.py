"""NVFP4 read copy -- the oracle.

TEST INFRASTRUCTURE (see the package docstring): never imported by the product.

The method keeps a high-precision checkpoint that drives the recurrence and a
low-precision copy that serves the reads; 4-bit NVFP4 reads are the case the
pages single out ([AT Pulse] §What happened, the quantization item, and
§Capabilities and access, the low-precision kernels; [Clarity] claim ledger
[15]; the NVIDIA blog summary under §Accuracy).  The pages give no block
layout, so the format comes from its public definition:

* elements are E2M1 (OCP Microscaling Formats v1.0): 1 sign bit, 2 exponent
  bits with bias 1, 1 mantissa bit; exponent field 0 encodes m * 0.5; the
  magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities or NaN; rounding to
  nearest, ties to the even code, saturating to +-6;
* every 16 consecutive elements share one E4M3 scale (oracle.fp8's encoder),
  and a float32 scale sits above the block scales (NVIDIA's two-level NVFP4).

Reading (the plainest one the pages leave open): the float32 second-level
scale is per (head, headdim row), the granularity of the FP8 copy's scale; a
block is 16 consecutive dstate columns of one row.  The block scale maps the
block's largest magnitude to the largest element code, 6, and the row scale
maps the row's largest magnitude to 6 * 448 = 2688.

Row quantiser, every step one correctly rounded float32 operation:

    amax  = max_n |h[n]|
    s_r   = fl32(amax / 2688)                     row scale (stored)
    k_r   = fl32(448 / amax)
    per block c of 16 columns, amax_c = max |h[n]| over the block:
      sb_c  = e4m3_rne_satfinite(fl32(amax_c * k_r))   block scale code (stored)
      d_c   = fl32(e4m3(sb_c) * s_r)
      inv_c = fl32(1 / d_c)
      code  = e2m1_rne_satfinite(fl32(h[n] * inv_c))
    value = e2m1(code) * e4m3(sb_c) * s_r     (exact; decoded in float64)

Guards: when amax == 0, s_r == 0 or k_r overflows, the row stores s_r = 0 and
k_r = 0 is used (so every block scale is 0); when d_c == 0 or inv_c overflows,
inv_c = 0.  A zero inv_c gives each code the sign of h[n] times zero (+-0).

Storage of one head (P rows, N columns): the codes ``[P][N/2]`` bytes, element
2i of a row in the low nibble of byte i and element 2i+1 in the high nibble,
followed by the block-scale codes ``[P][N/16]``; the row scales are a separate
``[P]`` float32 array.

fl32(a op b) is computed as float64 then rounded to float32; for one +, *, /
of float32 operands this double rounding is exact (53 >= 2*24 + 2).
"""
from __future__ import annotations

import numpy as np

from oracle.fp8 import e4m3_decode, e4m3_encode

E2M1_MAX = 6.0
ROW_TARGET = 6.0 * 448.0          # the row maximum maps here: largest element code x largest block scale
BLOCK = 16


def e2m1_encode(v) -> np.ndarray:
    """float32 values -> uint8 E2M1 codes 0..15 (RNE, satfinite; NaN -> +6)."""
    v = np.asarray(v, np.float32)
    a = np.abs(v.astype(np.float64))
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, 1e300))
    # spacing of the grid around a: 0.5 below 2 (subnormals and the binade
    # [1, 2) share it), else half the binade's lower end
    _, ex = np.frexp(a)                                # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, 0)                          # floor(log2 a), at least 0
    quantum = np.ldexp(0.5, e)
    val = np.rint(a / quantum) * quantum               # ties to the even multiple = even code
    val = np.minimum(val, E2M1_MAX)                    # satfinite
    # the code of a grid value: exponent field and mantissa bit
    sub = val < 1.0
    code_sub = np.rint(val / 0.5).astype(np.int64)     # 0 or 1
    _, ex2 = np.frexp(np.where(sub, 1.0, val))
    E = ex2 - 1                                        # 0..2 for 1..6
    mant = np.rint((np.where(sub, 1.0, val) / np.ldexp(1.0, E) - 1.0) * 2).astype(np.int64)
    code = np.where(sub, code_sub, ((E + 1) << 1) | mant)
    code = np.where(nan, 0x7, code)
    sign = np.where(nan, 0, np.signbit(v).astype(np.int64))
    return (code | (sign << 3)).astype(np.uint8)


def e2m1_decode(code) -> np.ndarray:
    """E2M1 codes 0..15 -> float64 values."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    s = np.where(c & 0x8, -1.0, 1.0)
    ef = (c >> 1) & 0x3
    m = c & 0x1
    val = np.where(ef == 0, m * 0.5, (1.0 + m / 2.0) * np.ldexp(1.0, ef - 1))
    return s * val


def _fl32(a) -> np.ndarray:
    return np.asarray(a, np.float64).astype(np.float32)


def quantize_rows(h) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """float32 [..., N] (N a multiple of 16) -> (codes uint8 [..., N] one code per
    element, block-scale codes uint8 [..., N/16], row scales float32 [...])."""
    h = np.asarray(h, np.float32)
    N = h.shape[-1]
    assert N % BLOCK == 0
    amax = np.max(np.abs(h), axis=-1).astype(np.float64)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        s_r = _fl32(amax / ROW_TARGET)
        k_r = _fl32(448.0 / amax)
    bad = ~(amax > 0) | ~(s_r > 0) | ~np.isfinite(k_r)
    s_r = np.where(bad, np.float32(0), s_r).astype(np.float32)
    k_r = np.where(bad, np.float32(0), k_r).astype(np.float32)

    hb = h.reshape(h.shape[:-1] + (N // BLOCK, BLOCK))
    amax_c = np.max(np.abs(hb), axis=-1).astype(np.float64)
    sb = e4m3_encode(_fl32(amax_c * k_r[..., None].astype(np.float64)))
    d = _fl32(e4m3_decode(sb) * s_r[..., None].astype(np.float64))
    with np.errstate(divide="ignore", over="ignore"):
        inv = _fl32(1.0 / d.astype(np.float64))
    inv = np.where((d == 0) | ~np.isfinite(inv), np.float32(0), inv).astype(np.float32)
    prod = _fl32(hb.astype(np.float64) * inv[..., None].astype(np.float64))
    codes = e2m1_encode(prod).reshape(h.shape)
    return codes, sb, s_r


def dequantize_rows(codes, sb, s_r) -> np.ndarray:
    """e2m1(code) * e4m3(sb) * s_r, exact in float64 ([..., N])."""
    codes = np.asarray(codes, np.uint8)
    N = codes.shape[-1]
    scale = e4m3_decode(sb) * np.asarray(s_r, np.float32).astype(np.float64)[..., None]     # [..., N/16]
    return e2m1_decode(codes) * np.repeat(scale, BLOCK, axis=-1).reshape(codes.shape[:-1] + (N,))


def pack_codes(codes) -> np.ndarray:
    """[..., N] codes -> [..., N/2] bytes: element 2i low nibble, 2i+1 high nibble."""
    c = np.asarray(codes, np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def head_copy(h) -> tuple[np.ndarray, np.ndarray]:
    """float32 [..., P, N] head tiles -> (the stored bytes [..., P*N/2 + P*N/16]:
    packed codes then block scales, row scales [..., P])."""
    h = np.asarray(h, np.float32)
    P, N = h.shape[-2], h.shape[-1]
    codes, sb, s_r = quantize_rows(h)
    lead = h.shape[:-2]
    packed = pack_codes(codes).reshape(lead + (P * N // 2,))
    return np.concatenate([packed, sb.reshape(lead + (P * N // BLOCK,))], axis=-1), s_r


def head_dequantize(stored, s_r, P: int, N: int) -> np.ndarray:
    """Inverse of head_copy: the float64 values the reads see, [..., P, N]."""
    stored = np.asarray(stored, np.uint8)
    lead = stored.shape[:-1]
    packed = stored[..., :P * N // 2].reshape(lead + (P, N // 2))
    sb = stored[..., P * N // 2:].reshape(lead + (P, N // BLOCK))
    return dequantize_rows(unpack_codes(packed), sb, s_r)
