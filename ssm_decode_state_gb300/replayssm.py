"""Python binding of libreplayssm.so (ctypes).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the C ABI.  PyTorch provides device memory and the current
stream.  If the library has not been built, importing this module raises.

Functions take torch tensors laid out as the C header states and return the
output tensor; a non-zero status raises ``ReplaySSMError``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libreplayssm.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libreplayssm.so is not built ({_LIB_PATH}); run "
                      "`python -c 'import __graft_entry__ as g; g.build()'`")
_lib = ctypes.CDLL(_LIB_PATH)

EXPORTS = [
    "replayssm_decode", "replayssm_decode_noalloc", "replayssm_flush", "replayssm_verify", "replayssm_rollback",
    "replayssm_requant", "replayssm_conventional_decode", "replayssm_conventional_verify",
    "replayssm_conventional_select", "replayssm_gdn_decode", "replayssm_gdn_flush", "replayssm_gdn_verify",
    "replayssm_gdn_rollback", "replayssm_gdn_conventional_decode", "replayssm_status_string", "replayssm_version",
    "replayssm_test_stalled_decode",
]

DEVERR_RING_META = 0x1
DEVERR_ROLLBACK = 0x2
DEVERR_SLOT = 0x4
DEVERR_TIMEOUT = 0x8


class ReplaySSMError(RuntimeError):
    pass


class Mamba2Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "nheads", "headdim", "dstate", "ngroups", "L", "read_copy", "io_bf16", "ckpt_f16")]


class Mamba2CacheC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("ckpt", "ckpt_q", "ckpt_scale", "rec_dt", "rec_x", "rec_B", "rec_C",
                 "ring_head", "ring_len", "arrive", "A", "D", "err", "slots")] + \
        [("capacity", ctypes.c_int32), ("sr_seed", ctypes.c_uint64)]


class GDNDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("batch", "nheads", "dk", "dv", "L")]


class GDNCacheC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("ckpt", "rec_k", "rec_v", "rec_alpha", "rec_beta", "ring_head", "ring_len",
                 "arrive", "err", "slots")] + [("capacity", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_sig = {
    "replayssm_decode": [_P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_decode_noalloc": [_P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_test_stalled_decode": [_P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_flush": [_P, _P, _P, _P],
    "replayssm_verify": [_P, _P, _I, _P, _P, _P, _P, _P, _P],
    "replayssm_rollback": [_P, _P, _I, _P, _P],
    "replayssm_requant": [_P, _P, _P],
    "replayssm_conventional_decode": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_conventional_verify": [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_conventional_select": [_I, _P, _I, _P, _P, _P],
    "replayssm_gdn_decode": [_P, _P, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_gdn_flush": [_P, _P, _P, _P],
    "replayssm_gdn_verify": [_P, _P, _I, _P, _P, _P, _P, _P, _P, _P],
    "replayssm_gdn_rollback": [_P, _P, _I, _P, _P],
    "replayssm_gdn_conventional_decode": [_P, _P, _P, _P, _P, _P, _P, _P, _P],
}
for _name, _args in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.replayssm_status_string.argtypes = [ctypes.c_int]
_lib.replayssm_status_string.restype = ctypes.c_char_p
_lib.replayssm_version.argtypes = []
_lib.replayssm_version.restype = ctypes.c_uint32


def library_path() -> str:
    return _LIB_PATH


def version() -> int:
    return int(_lib.replayssm_version())


def status_string(code: int) -> str:
    return _lib.replayssm_status_string(code).decode()


def _check(code: int) -> None:
    if code != 0:
        raise ReplaySSMError(f"replayssm status {code}: {status_string(code)}")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# --------------------------------------------------------------------- Mamba-2

@dataclass
class Mamba2Cache:
    """Device buffers of a Mamba-2 replay cache (caller-owned, as the ABI says)."""
    dims: Mamba2Dims
    ckpt: torch.Tensor
    ckpt_q: torch.Tensor | None
    ckpt_scale: torch.Tensor | None
    rec_dt: torch.Tensor
    rec_x: torch.Tensor
    rec_B: torch.Tensor
    rec_C: torch.Tensor | None
    ring_head: torch.Tensor
    ring_len: torch.Tensor
    arrive: torch.Tensor
    A: torch.Tensor
    D: torch.Tensor
    err: torch.Tensor
    slots: torch.Tensor | None = None      # [batch] int32 cache slot of each batch row (None: row b -> slot b)
    capacity: int = 0                      # sequences the cache holds (0: batch)
    sr_seed: int = 0                       # seed of the next call's stochastic rounding (FP16 checkpoint)

    def c_struct(self, slots=None) -> Mamba2CacheC:
        """The C struct; ``slots`` (int32 [batch] on the device) overrides the cache's map."""
        sl = self.slots if slots is None else slots
        vals = [_ptr(getattr(self, f)) for f, _ in Mamba2CacheC._fields_[:-3]]
        return Mamba2CacheC(*vals, _ptr(sl), int(self.capacity), int(self.sr_seed) & (2 ** 64 - 1))

    def _seeded(self, slots=None) -> Mamba2CacheC:
        """The C struct of a call that may flush: it takes the current seed and
        the next such call the following one."""
        cs = self.c_struct(slots)
        self.sr_seed = (int(self.sr_seed) + 1) & (2 ** 64 - 1)
        return cs


def mamba2_dims(batch, nheads, headdim, dstate, ngroups, L=16, read_copy=0, io_bf16=True,
                ckpt_f16=False) -> Mamba2Dims:
    return Mamba2Dims(batch, nheads, headdim, dstate, ngroups, L, int(read_copy), int(bool(io_bf16)),
                      int(bool(ckpt_f16)))


def mamba2_cache(dims: Mamba2Dims, A: torch.Tensor, D: torch.Tensor, ckpt: torch.Tensor | None = None,
                 keep_C: bool = True, device="cuda", capacity: int = 0) -> Mamba2Cache:
    """Allocate an empty-ring cache for ``capacity`` sequences (0: dims.batch).
    ``ckpt`` (if given) is used as the checkpoint."""
    H, P, N, G, L = dims.nheads, dims.headdim, dims.dstate, dims.ngroups, dims.L
    b = capacity if capacity > 0 else dims.batch
    io = torch.bfloat16 if dims.io_bf16 else torch.float32
    z = lambda *s, dtype=torch.float32: torch.zeros(*s, dtype=dtype, device=device)  # noqa: E731
    if ckpt is None:
        ckpt = z(b, H, P, N, dtype=torch.float16 if dims.ckpt_f16 else torch.float32)
    return Mamba2Cache(
        dims=dims, ckpt=ckpt,
        ckpt_q=(z(b, H, P, N, dtype=torch.uint8) if dims.read_copy == 1 else
                z(b, H, P * N // 2 + P * N // 16, dtype=torch.uint8) if dims.read_copy == 2 else None),
        ckpt_scale=z(b, H, P) if dims.read_copy else None,
        rec_dt=z(b, H, L), rec_x=z(b, H, L, P, dtype=io), rec_B=z(b, G, L, N, dtype=io),
        rec_C=z(b, G, L, N, dtype=io) if keep_C else None,
        ring_head=z(b, dtype=torch.int32), ring_len=z(b, dtype=torch.int32),
        arrive=z(b, dtype=torch.int32),
        A=A.to(device=device, dtype=torch.float32).contiguous(),
        D=D.to(device=device, dtype=torch.float32).contiguous(),
        err=z(1, dtype=torch.int32), capacity=int(capacity))


def decode(cache: Mamba2Cache, dt, x, B, C, y=None, stream=None, slots=None) -> torch.Tensor:
    d = cache.dims
    if y is None:
        y = torch.empty(d.batch, d.nheads, d.headdim, dtype=torch.float32, device=dt.device)
    cs = cache._seeded(slots)
    _check(_lib.replayssm_decode(ctypes.byref(d), ctypes.byref(cs), _ptr(dt), _ptr(x), _ptr(B), _ptr(C),
                                 _ptr(y), _stream(stream)))
    return y


def decode_noalloc(cache: Mamba2Cache, dt, x, B, C, y=None, stream=None, slots=None) -> torch.Tensor:
    """decode() for callers that cannot allocate: the arrival counters live in
    the library's own device memory (cache.arrive is not used; batch <= 4096)."""
    d = cache.dims
    if y is None:
        y = torch.empty(d.batch, d.nheads, d.headdim, dtype=torch.float32, device=dt.device)
    cs = cache._seeded(slots)
    cs.arrive = None
    _check(_lib.replayssm_decode_noalloc(ctypes.byref(d), ctypes.byref(cs), _ptr(dt), _ptr(x), _ptr(B),
                                         _ptr(C), _ptr(y), _stream(stream)))
    return y


def stalled_decode(cache: Mamba2Cache, dt, x, B, C, y=None, stream=None) -> torch.Tensor:
    """The bounded-wait test hook (replayssm_test_stalled_decode): a decode whose
    first wait runs out; the cache is not usable afterwards."""
    d = cache.dims
    if y is None:
        y = torch.empty(d.batch, d.nheads, d.headdim, dtype=torch.float32, device=dt.device)
    cs = cache._seeded()
    _check(_lib.replayssm_test_stalled_decode(ctypes.byref(d), ctypes.byref(cs), _ptr(dt), _ptr(x), _ptr(B),
                                              _ptr(C), _ptr(y), _stream(stream)))
    return y


def flush(cache: Mamba2Cache, mask=None, stream=None, slots=None) -> None:
    cs = cache._seeded(slots)
    _check(_lib.replayssm_flush(ctypes.byref(cache.dims), ctypes.byref(cs), _ptr(mask), _stream(stream)))


def verify(cache: Mamba2Cache, dt, x, B, C, y=None, stream=None, slots=None) -> torch.Tensor:
    d = cache.dims
    T = dt.shape[1]
    if y is None:
        y = torch.empty(d.batch, T, d.nheads, d.headdim, dtype=torch.float32, device=dt.device)
    cs = cache._seeded(slots)
    _check(_lib.replayssm_verify(ctypes.byref(d), ctypes.byref(cs), T, _ptr(dt), _ptr(x), _ptr(B), _ptr(C),
                                 _ptr(y), _stream(stream)))
    return y


def rollback(cache: Mamba2Cache, T: int, accepted, stream=None, slots=None) -> None:
    cs = cache.c_struct(slots)
    _check(_lib.replayssm_rollback(ctypes.byref(cache.dims), ctypes.byref(cs), T, _ptr(accepted),
                                   _stream(stream)))


def requant(cache: Mamba2Cache, stream=None) -> None:
    cs = cache.c_struct()
    _check(_lib.replayssm_requant(ctypes.byref(cache.dims), ctypes.byref(cs), _stream(stream)))


def conventional_decode(dims: Mamba2Dims, state, A, D, dt, x, B, C, y=None, stream=None) -> torch.Tensor:
    if y is None:
        y = torch.empty(dims.batch, dims.nheads, dims.headdim, dtype=torch.float32, device=dt.device)
    _check(_lib.replayssm_conventional_decode(ctypes.byref(dims), _ptr(state), _ptr(A), _ptr(D), _ptr(dt),
                                              _ptr(x), _ptr(B), _ptr(C), _ptr(y), _stream(stream)))
    return y


def conventional_verify(dims: Mamba2Dims, pool, slot, A, D, dt, x, B, C, err, y=None,
                        stream=None) -> torch.Tensor:
    T = dt.shape[1]
    if y is None:
        y = torch.empty(dims.batch, T, dims.nheads, dims.headdim, dtype=torch.float32, device=dt.device)
    _check(_lib.replayssm_conventional_verify(ctypes.byref(dims), _ptr(pool), _ptr(slot), T, _ptr(A), _ptr(D),
                                              _ptr(dt), _ptr(x), _ptr(B), _ptr(C), _ptr(y), _ptr(err),
                                              _stream(stream)))
    return y


def conventional_select(slot, T: int, accepted, err, stream=None) -> None:
    _check(_lib.replayssm_conventional_select(slot.shape[0], _ptr(slot), T, _ptr(accepted), _ptr(err),
                                              _stream(stream)))


# ------------------------------------------------------------------------ GDN

@dataclass
class GDNCache:
    dims: GDNDims
    ckpt: torch.Tensor
    rec_k: torch.Tensor
    rec_v: torch.Tensor
    rec_alpha: torch.Tensor
    rec_beta: torch.Tensor
    ring_head: torch.Tensor
    ring_len: torch.Tensor
    arrive: torch.Tensor
    err: torch.Tensor
    slots: torch.Tensor | None = None      # [batch] int32 cache slot of each batch row (None: row b -> slot b)
    capacity: int = 0                      # sequences the cache holds (0: batch)

    def c_struct(self, slots=None) -> GDNCacheC:
        """The C struct; ``slots`` (int32 [batch] on the device) overrides the cache's map."""
        sl = self.slots if slots is None else slots
        vals = [_ptr(getattr(self, f)) for f, _ in GDNCacheC._fields_[:-2]]
        return GDNCacheC(*vals, _ptr(sl), int(self.capacity))


def gdn_dims(batch, nheads, dk, dv, L=16) -> GDNDims:
    return GDNDims(batch, nheads, dk, dv, L)


def gdn_cache(dims: GDNDims, ckpt=None, device="cuda", capacity: int = 0) -> GDNCache:
    """Allocate an empty-ring cache for ``capacity`` sequences (0: dims.batch)."""
    H, dk, dv, L = dims.nheads, dims.dk, dims.dv, dims.L
    b = capacity if capacity > 0 else dims.batch
    z = lambda *s, dtype=torch.float32: torch.zeros(*s, dtype=dtype, device=device)  # noqa: E731
    if ckpt is None:
        ckpt = z(b, H, dv, dk)
    return GDNCache(dims=dims, ckpt=ckpt, rec_k=z(b, H, L, dk, dtype=torch.bfloat16),
                    rec_v=z(b, H, L, dv, dtype=torch.bfloat16), rec_alpha=z(b, H, L), rec_beta=z(b, H, L),
                    ring_head=z(b, dtype=torch.int32), ring_len=z(b, dtype=torch.int32),
                    arrive=z(b, dtype=torch.int32), err=z(1, dtype=torch.int32), capacity=int(capacity))


def gdn_decode(cache: GDNCache, q, k, v, alpha, beta, o=None, stream=None, slots=None) -> torch.Tensor:
    d = cache.dims
    if o is None:
        o = torch.empty(d.batch, d.nheads, d.dv, dtype=torch.float32, device=q.device)
    cs = cache.c_struct(slots)
    _check(_lib.replayssm_gdn_decode(ctypes.byref(d), ctypes.byref(cs), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                     _ptr(beta), _ptr(o), _stream(stream)))
    return o


def gdn_flush(cache: GDNCache, mask=None, stream=None, slots=None) -> None:
    cs = cache.c_struct(slots)
    _check(_lib.replayssm_gdn_flush(ctypes.byref(cache.dims), ctypes.byref(cs), _ptr(mask), _stream(stream)))


def gdn_verify(cache: GDNCache, q, k, v, alpha, beta, o=None, stream=None, slots=None) -> torch.Tensor:
    """Score T drafts per sequence (q, k [b, T, H, dk], v [b, T, H, dv], alpha, beta
    [b, T, H]); returns o [b, T, H, dv].  Appends the drafts' records."""
    d = cache.dims
    T = alpha.shape[1]
    if o is None:
        o = torch.empty(d.batch, T, d.nheads, d.dv, dtype=torch.float32, device=q.device)
    cs = cache.c_struct(slots)
    _check(_lib.replayssm_gdn_verify(ctypes.byref(d), ctypes.byref(cs), T, _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(alpha), _ptr(beta), _ptr(o), _stream(stream)))
    return o


def gdn_rollback(cache: GDNCache, T: int, accepted, stream=None, slots=None) -> None:
    """Keep accepted[b] of the T drafts of the last verify (int32 device tensor)."""
    cs = cache.c_struct(slots)
    _check(_lib.replayssm_gdn_rollback(ctypes.byref(cache.dims), ctypes.byref(cs), T, _ptr(accepted),
                                       _stream(stream)))


def gdn_conventional_decode(dims: GDNDims, state, q, k, v, alpha, beta, o=None, stream=None) -> torch.Tensor:
    if o is None:
        o = torch.empty(dims.batch, dims.nheads, dims.dv, dtype=torch.float32, device=q.device)
    _check(_lib.replayssm_gdn_conventional_decode(ctypes.byref(dims), _ptr(state), _ptr(q), _ptr(k), _ptr(v),
                                                  _ptr(alpha), _ptr(beta), _ptr(o), _stream(stream)))
    return o
