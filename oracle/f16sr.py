"""FP16 checkpoint recurrence with stochastic rounding -- the oracle.

TEST INFRASTRUCTURE (see the package docstring): never imported by the product.

The pages pair low-precision state reads with an FP16 (stochastic rounding)
or FP8 recurrence ([AT Pulse] §Capabilities and access, the low-precision
kernels; the NVIDIA blog summary under §Accuracy).  Reading taken here: the
checkpoint itself is stored in FP16; between flushes nothing rounds it (the
buffered records carry the new tokens in their own precision); at every flush
the folded state, computed at higher precision and then held as float32, is
rounded to FP16 stochastically, so the expected rounding error is zero and
does not build up over flushes.  The pages give no rounding recipe or random
source, so both are fixed here:

Stochastic rounding of a float32 v with a 16-bit random integer r:
    a  = |v|; if a >= 65504 the result is +-65504 (largest finite FP16)
    lo = the largest FP16 value <= a
    u  = spacing of FP16 above lo: 2^-24 below 2^-14, else 2^(floor(log2 lo) - 10)
    p  = (a - lo) / u                     (in [0, 1), exact)
    result = sign(v) * (lo + u if r < p * 65536 else lo)
For a normal FP16 result p is a multiple of 2^-13, so P(round up) = p exactly
and the rounding is unbiased; below 2^-14 the bias is under 2^-16 of a step.

Random integers: Philox4x32-10, the counter-based generator of Salmon, Moraes,
Dror and Shaw ("Parallel random numbers: as easy as 1, 2, 3", SC'11): a 128-bit
counter and a 64-bit key, ten rounds of two 32x32 -> 64-bit multiplications by
0xD2511F53 and 0xCD9E8D57 with the key advanced by the Weyl increments
0x9E3779B9 and 0xBB67AE85 between rounds.  One generator call serves 8
consecutive columns: the element in column n, row p of head h of cache slot s
at a call with seed S takes
    out = Philox4x32-10(counter = (n / 8, p, h, s), key = (S mod 2^32, S / 2^32))
    r   = 16-bit half (n mod 2) of word ((n mod 8) / 2) of out  (low half first).

The recurrence: the Mamba-2 stepwise update of oracle.mamba2, in float64, from
an FP16 checkpoint; a flush (the step at which a sequence's ring of L records
fills) replaces the state by SR_16(fl32(state)).
"""
from __future__ import annotations

import numpy as np

from oracle.mamba2 import Mamba2Stepwise

_M0, _M1 = 0xD2511F53, 0xCD9E8D57
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
F16_MAX = 65504.0


def philox4x32_10(ctr, key) -> np.ndarray:
    """ctr uint32 [..., 4], key uint32 [..., 2] (broadcast) -> uint32 [..., 4]."""
    c = np.asarray(ctr, np.uint64) & 0xFFFFFFFF
    k = np.asarray(key, np.uint64) & 0xFFFFFFFF
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0, k1 = k[..., 0], k[..., 1]
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + _W0) & 0xFFFFFFFF
            k1 = (k1 + _W1) & 0xFFFFFFFF
        p0 = c0 * np.uint64(_M0)                  # < 2^64: exact in uint64
        p1 = c2 * np.uint64(_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(0xFFFFFFFF)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(0xFFFFFFFF)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def random16(seed: int, slot: int, head: int, P: int, N: int) -> np.ndarray:
    """The 16-bit random integers of one head's P x N elements (uint32 [P, N])."""
    ctr = np.zeros((P, N // 8, 4), np.uint64)
    ctr[..., 0] = np.arange(N // 8)[None, :]
    ctr[..., 1] = np.arange(P)[:, None]
    ctr[..., 2] = head
    ctr[..., 3] = slot
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], np.uint64)
    out = philox4x32_10(ctr, key).astype(np.uint64)          # [P, N/8, 4]
    n = np.arange(N)
    word = out[:, n // 8, (n % 8) // 2]                      # [P, N]
    return ((word >> (16 * (n % 2)).astype(np.uint64)) & 0xFFFF).astype(np.uint32)


def _f16_rz(a: np.ndarray) -> np.ndarray:
    """Largest FP16 value <= a (a >= 0, float64 array), as float64."""
    r = a.astype(np.float16)                                 # round to nearest even
    r = np.where(r.astype(np.float64) > a, np.nextafter(r, np.float16(0)), r)
    return r.astype(np.float64)


def sr_f16(v, r) -> np.ndarray:
    """Stochastic rounding of float32 values v with 16-bit random integers r
    (same shape) -> float16."""
    v = np.asarray(v, np.float32)
    a = np.abs(v.astype(np.float64))
    lo = _f16_rz(np.minimum(a, F16_MAX))
    e = np.floor(np.log2(np.where(lo > 0, lo, 1.0)))
    u = np.where(lo < 2.0 ** -14, 2.0 ** -24, np.ldexp(1.0, (e - 10).astype(np.int64)))
    p = (a - lo) / u
    up = np.asarray(r, np.float64) < p * 65536.0
    res = np.where(a >= F16_MAX, F16_MAX, lo + np.where(up, u, 0.0))
    return (np.where(np.signbit(v), -res, res)).astype(np.float16)


class Mamba2F16SR(Mamba2Stepwise):
    """Stepwise Mamba-2 recurrence from an FP16 checkpoint, with the state
    rounded stochastically to FP16 whenever a sequence's ring of L records
    fills (every L-th decode token from an empty ring)."""

    def __init__(self, A, D, ngroups: int, h0_f16, L: int, slots=None, ring_len=None):
        super().__init__(A, D, ngroups, np.asarray(h0_f16, np.float16).astype(np.float64))
        self.L = L
        b = self.h.shape[0]
        self.slots = np.arange(b) if slots is None else np.asarray(slots)
        self.len = np.zeros(b, np.int64) if ring_len is None else np.asarray(ring_len, np.int64).copy()

    def fold(self, b: int, seed: int) -> None:
        """The flush of sequence (row) b: SR_16(fl32(state)) with the call's seed."""
        H, P, N = self.h.shape[1:]
        v = self.h[b].astype(np.float32)
        out = np.empty((H, P, N), np.float16)
        for h in range(H):
            out[h] = sr_f16(v[h], random16(seed, int(self.slots[b]), h, P, N))
        self.h[b] = out.astype(np.float64)
        self.len[b] = 0

    def decode(self, dt, x, B, C, seed: int) -> np.ndarray:
        """One token per sequence; the sequences whose ring fills fold."""
        y = self.step(dt, x, B, C)
        for b in range(self.h.shape[0]):
            if self.len[b] + 1 >= self.L:
                self.fold(b, seed)
            else:
                self.len[b] += 1
        return y
