"""Algorithmic HBM bytes of each decode path, per sequence and step.

Only the bytes the method must move are counted: the checkpoint (or its read
copy) read once, written only when folded; the token inputs read once; the
output written once; the new record written once; each buffered record read
once.  The pages' size arithmetic is the unit check of this model: a 4 MiB
FP32 state per sequence and layer equals the KV cache of 8,192 tokens at
0.5 KiB per token; with five SSM layers per attention layer that is 40,960
tokens, and a load plus a store every step 81,920 (Clarity, key figures and
claim ledger [10], [11], [19]-[21]).  Replay keeps the checkpoint reads and
drops most of the writes, which roughly halves the state traffic (AT Pulse
§What happened).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Mamba2Units:
    S: int    # FP32 checkpoint
    Sq: int   # FP8 read copy: codes + one float32 scale per row
    Sq4: int  # NVFP4 read copy: 4-bit codes + an E4M3 scale per 16 columns + a float32 scale per row
    I: int    # one token's inputs: dt, x, B, C
    Y: int    # one token's output y (float32)
    Rw: int   # one record written: dt, x, B, C
    Rr: int   # one buffered record read: dt, x, B (C is never read back)


def mamba2_units(nheads, headdim, dstate, ngroups, io_bytes=2, keep_C=True) -> Mamba2Units:
    H, P, N, G = nheads, headdim, dstate, ngroups
    S = H * P * N * 4
    Sq = H * P * N + H * P * 4
    Sq4 = H * P * N // 2 + H * P * N // 16 + H * P * 4
    I = H * 4 + H * P * io_bytes + 2 * G * N * io_bytes
    Y = H * P * 4
    Rw = H * 4 + H * P * io_bytes + (2 if keep_C else 1) * G * N * io_bytes
    Rr = H * 4 + H * P * io_bytes + G * N * io_bytes
    return Mamba2Units(S, Sq, Sq4, I, Y, Rw, Rr)


def mamba2_conventional(u: Mamba2Units) -> int:
    return 2 * u.S + u.I + u.Y


def _copy_bytes(u: Mamba2Units, read_copy) -> int:
    """Size of the read copy: none (0 / False), FP8 (1 / True), NVFP4 (2)."""
    return {0: 0, 1: u.Sq, 2: u.Sq4}[int(read_copy)]


def mamba2_replay_decode(u: Mamba2Units, len_before: int, L: int, read_copy: int = 0,
                         ckpt_f16: bool = False) -> int:
    """One replay decode step of a sequence holding ``len_before`` records; a
    read copy (1 FP8, 2 NVFP4) replaces the checkpoint read on non-flush steps
    and is rewritten at the flush; an FP16 checkpoint is half the bytes."""
    fold = len_before + 1 >= L
    S = u.S // 2 if ckpt_f16 else u.S
    b = u.I + u.Y + len_before * u.Rr
    if fold:
        b += 2 * S + _copy_bytes(u, read_copy)
    else:
        b += (_copy_bytes(u, read_copy) or S) + u.Rw
    return b


def mamba2_replay_period(u: Mamba2Units, L: int, read_copy: int = 0, ckpt_f16: bool = False) -> float:
    """Mean over one flush period of L steps from an empty ring."""
    return sum(mamba2_replay_decode(u, k, L, read_copy, ckpt_f16) for k in range(L)) / L


def mamba2_verify(u: Mamba2Units, len_before: int, T: int, L: int) -> int:
    pre = len_before + T > L
    return u.S + (u.S if pre else 0) + T * (u.I + u.Y + u.Rw) + len_before * u.Rr


def mamba2_conventional_verify(u: Mamba2Units, T: int) -> int:
    return u.S + T * u.S + T * (u.I + u.Y)


@dataclass(frozen=True)
class GDNUnits:
    S: int
    I: int
    Y: int
    Rw: int
    Rr: int


def gdn_units(nheads, dk, dv) -> GDNUnits:
    H = nheads
    S = H * dv * dk * 4
    I = 2 * H * dk * 2 + H * dv * 2 + 2 * H * 4
    Y = H * dv * 4
    R = H * dk * 2 + H * dv * 2 + 2 * H * 4
    return GDNUnits(S, I, Y, R, R)


def gdn_conventional(u: GDNUnits) -> int:
    return 2 * u.S + u.I + u.Y


def gdn_replay_decode(u: GDNUnits, len_before: int, L: int) -> int:
    fold = len_before + 1 >= L
    b = u.I + u.Y + len_before * u.Rr
    return b + (2 * u.S if fold else u.S + u.Rw)


def gdn_replay_period(u: GDNUnits, L: int) -> float:
    return sum(gdn_replay_decode(u, k, L) for k in range(L)) / L


def gdn_verify(u: GDNUnits, len_before: int, T: int, L: int) -> int:
    """Replay verify of T drafts: the checkpoint once (written back on a pre-flush),
    the T drafts' inputs and outputs, their records appended, the buffered records read."""
    pre = len_before + T > L
    return u.S + (u.S if pre else 0) + T * (u.I + u.Y + u.Rw) + len_before * u.Rr


def mamba2_cache_bytes(nheads, headdim, dstate, ngroups, L, io_bytes=2, keep_C=True,
                       read_copy: int = 0, ckpt_f16: bool = False) -> dict:
    """Device memory one sequence's replay cache holds per layer, by part: the
    checkpoint, the read copy, the ring of L records and its pointers.  Engines
    that cap concurrent requests by state memory now hold the record buffer
    beside each checkpoint, so their accounting changes with it (AT Pulse,
    cost item); the conventional state is the checkpoint alone."""
    H, P, N, G = nheads, headdim, dstate, ngroups
    u = mamba2_units(H, P, N, G, io_bytes, keep_C)
    ckpt = u.S // 2 if ckpt_f16 else u.S
    ring = L * (H * 4 + H * P * io_bytes + (2 if keep_C else 1) * G * N * io_bytes)
    parts = {"checkpoint": ckpt, "read_copy": _copy_bytes(u, read_copy), "ring": ring, "pointers": 12}
    parts["total"] = sum(parts.values())
    parts["conventional"] = u.S
    return parts


def sequences_that_fit(budget_bytes: int, layers: int, **cache_kw) -> dict:
    """Concurrent sequences a device-memory budget holds for `layers` SSM layers,
    replay cache against conventional state."""
    c = mamba2_cache_bytes(**cache_kw)
    return {"replay": budget_bytes // (layers * c["total"]), "conventional": budget_bytes // (layers * c["conventional"])}
