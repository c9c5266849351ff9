"""FP8 E4M3 read copy -- the oracle.

TEST INFRASTRUCTURE (see the package docstring): never imported by the product.

The method keeps a high-precision checkpoint that drives the recurrence and a
low-precision copy that serves reads, so read rounding does not compound
([AT Pulse] §What happened and §Technical analysis, quantization; [Clarity]
claim ledger [15]).  The pages name FP8 among the low-precision formats
([AT Pulse] §Capabilities and access) but give no scaling scheme.  Reading:
one float32 scale per (head, headdim row) of the checkpoint, re-quantised at
every flush.

Encoder written from the OCP 8-bit floating point definition of E4M3 (the
"fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
exponent field 0 encodes subnormals m/8 * 2^-6; no infinities; S.1111.111 is
NaN; largest finite magnitude 1.75 * 2^8 = 448.  Rounding is to nearest, ties
to even, saturating to +-448 ("satfinite"); NaN stays NaN.

Row quantiser, every step one correctly-rounded float32 operation:

    amax  = max_n |h[n]|
    scale = fl32(amax / 448)
    inv   = fl32(448 / amax)
    code  = e4m3_rne_satfinite(fl32(h[n] * inv))
    value = fl32(e4m3(code) * scale)

A row with amax == 0, or whose inv overflows float32, is stored as zero codes
with scale 1.  fl32(a op b) is computed as float64 then rounded to float32;
for a single +, *, / of float32 operands this double rounding is exact
(53 >= 2*24 + 2), so it equals the float32 operation rounded once.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_encode(v) -> np.ndarray:
    """float32 values -> uint8 E4M3 codes (RNE, satfinite)."""
    v = np.asarray(v, np.float32)
    a = np.abs(v.astype(np.float64))
    sign = np.signbit(v).astype(np.uint8) << 7
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, 1e300))

    # exponent of a's binade, floor(log2 a), but never below the smallest
    # normal exponent -6: below it the spacing stays 2^-9 (subnormals)
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, -6)
    quantum = np.ldexp(1.0, e - 3)                 # 3 mantissa bits
    val = np.rint(a / quantum) * quantum           # ties to even
    val = np.minimum(val, E4M3_MAX)                # satfinite

    code = np.zeros(v.shape, np.uint8)
    sub = val < 2.0 ** -6
    code_sub = np.rint(val / 2.0 ** -9).astype(np.int64)
    _, ex2 = np.frexp(np.where(sub, 1.0, val))
    E = ex2 - 1
    mant = np.rint((np.where(sub, 1.0, val) / np.ldexp(1.0, E) - 1.0) * 8).astype(np.int64)
    code_norm = ((E + 7) << 3) | mant
    code = np.where(sub, code_sub, code_norm).astype(np.uint8)
    code = np.where(nan, np.uint8(0x7F), code).astype(np.uint8)
    return (code | sign).astype(np.uint8)


def e4m3_decode(code) -> np.ndarray:
    """uint8 E4M3 codes -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ef == 0, m / 8.0 * 2.0 ** -6,
                   (1.0 + m / 8.0) * np.ldexp(1.0, ef - 7))
    val = np.where((ef == 0xF) & (m == 0x7), np.nan, val)
    return s * val


def _fl32(a) -> np.ndarray:
    return np.asarray(a, np.float64).astype(np.float32)


def quantize_rows(h) -> tuple[np.ndarray, np.ndarray]:
    """float32 [..., N] -> (codes uint8 [..., N], scale float32 [...])."""
    h = np.asarray(h, np.float32)
    amax = np.max(np.abs(h), axis=-1)
    with np.errstate(divide="ignore", over="ignore"):
        inv = _fl32(448.0 / amax.astype(np.float64))
        scale = _fl32(amax.astype(np.float64) / 448.0)
    bad = (amax == 0) | ~np.isfinite(inv)
    inv = np.where(bad, np.float32(0), inv).astype(np.float32)
    scale = np.where(bad, np.float32(1), scale).astype(np.float32)
    prod = _fl32(h.astype(np.float64) * inv[..., None].astype(np.float64))
    return e4m3_encode(prod), scale


def dequantize_rows(codes, scale) -> np.ndarray:
    """fl32(e4m3(code) * scale) as float32."""
    return _fl32(e4m3_decode(codes) * np.asarray(scale, np.float32)[..., None].astype(np.float64))
