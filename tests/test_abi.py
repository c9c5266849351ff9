"""The C ABI: the library builds, loads, exports every declared entry point,
its structs match the binding, and host-side argument checks return their
status before anything is launched (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "replayssm.h")


@pytest.fixture(scope="module")
def rs():
    import __graft_entry__
    __graft_entry__.build()
    from ssm_decode_state_gb300 import replayssm
    return replayssm


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(replayssm_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(rs):
    lib = ctypes.CDLL(rs.library_path())
    declared = _declared()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(rs.EXPORTS) == declared


def test_struct_layout_matches_binding(rs, tmp_path):
    """Compile a C probe against the header and compare sizes/offsets."""
    probe = tmp_path / "probe.c"
    probe.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "replayssm.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(rssm_mamba2_dims), sizeof(rssm_mamba2_cache),
         sizeof(rssm_gdn_dims), sizeof(rssm_gdn_cache), offsetof(rssm_mamba2_cache, err),
         offsetof(rssm_mamba2_cache, arrive), offsetof(rssm_gdn_cache, err),
         offsetof(rssm_mamba2_cache, capacity), offsetof(rssm_mamba2_cache, sr_seed),
         offsetof(rssm_mamba2_dims, ckpt_f16));
  return 0;
}''')
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(probe), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert out == [ctypes.sizeof(rs.Mamba2Dims), ctypes.sizeof(rs.Mamba2CacheC),
                   ctypes.sizeof(rs.GDNDims), ctypes.sizeof(rs.GDNCacheC),
                   rs.Mamba2CacheC.err.offset, rs.Mamba2CacheC.arrive.offset, rs.GDNCacheC.err.offset,
                   rs.Mamba2CacheC.capacity.offset, rs.Mamba2CacheC.sr_seed.offset, rs.Mamba2Dims.ckpt_f16.offset]


def test_status_strings(rs):
    for code in range(7):
        assert rs.status_string(code)
    assert rs.version() == 0x100


# ---- host-side argument checks (each returns before any launch)

FAKE = 0x10000          # 16-byte aligned, never dereferenced: every case fails first
MIS = 0x10008


def _m2(rs, **kw):
    d = dict(batch=2, nheads=4, headdim=16, dstate=16, ngroups=1, L=16, read_copy=0, io_bf16=1, ckpt_f16=0)
    d.update(kw)
    return rs.Mamba2Dims(**d)


def _cache(rs, **kw):
    c = {f: FAKE for f, _ in rs.Mamba2CacheC._fields_}
    c.update(kw)
    return rs.Mamba2CacheC(**c)


def _decode(rs, dims, cache, x=FAKE):
    lib = rs._lib
    return lib.replayssm_decode(ctypes.byref(dims) if dims is not None else None,
                                ctypes.byref(cache), FAKE, x, FAKE, FAKE, FAKE, None)


def test_null_and_shape_errors(rs):
    assert _decode(rs, None, _cache(rs)) == 1
    assert _decode(rs, _m2(rs, batch=0), _cache(rs)) == 3          # empty batch: rejected, nothing enqueued
    assert _decode(rs, _m2(rs, dstate=48), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, headdim=12), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, nheads=6, ngroups=4), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, L=0), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, L=33), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, read_copy=3), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, ckpt_f16=2), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, read_copy=-1), _cache(rs)) == 3
    assert _decode(rs, _m2(rs, read_copy=2), _cache(rs, ckpt_q=None)) == 1   # NVFP4 copy missing
    assert _decode(rs, _m2(rs), _cache(rs, ring_len=None)) == 1
    assert _decode(rs, _m2(rs), _cache(rs, arrive=None)) == 1
    assert _decode(rs, _m2(rs, read_copy=1), _cache(rs, ckpt_q=None)) == 1


def test_alignment_errors(rs):
    assert _decode(rs, _m2(rs), _cache(rs, ckpt=MIS)) == 2
    assert _decode(rs, _m2(rs), _cache(rs, rec_x=MIS)) == 2
    assert _decode(rs, _m2(rs), _cache(rs), x=MIS) == 2


def test_verify_draft_count(rs):
    lib = rs._lib
    d, c = _m2(rs, L=4), _cache(rs)
    for T in (0, 5, 9):
        assert lib.replayssm_verify(ctypes.byref(d), ctypes.byref(c), T, FAKE, FAKE, FAKE, FAKE,
                                    FAKE, None) == 4
    assert lib.replayssm_rollback(ctypes.byref(d), ctypes.byref(c), 0, FAKE, None) == 4
    assert lib.replayssm_conventional_select(4, FAKE, 9, FAKE, FAKE, None) == 4
    assert lib.replayssm_conventional_select(0, FAKE, 2, FAKE, FAKE, None) == 3


def test_gdn_checks(rs):
    lib = rs._lib
    c = rs.GDNCacheC(**{f: FAKE for f, _ in rs.GDNCacheC._fields_})
    bad = [rs.GDNDims(2, 4, 48, 64, 16), rs.GDNDims(2, 4, 64, 12, 16), rs.GDNDims(0, 4, 64, 64, 16)]
    for d in bad:
        assert lib.replayssm_gdn_decode(ctypes.byref(d), ctypes.byref(c), FAKE, FAKE, FAKE, FAKE,
                                        FAKE, FAKE, None) == 3
    d = rs.GDNDims(2, 4, 64, 64, 16)
    c2 = rs.GDNCacheC(**{**{f: FAKE for f, _ in rs.GDNCacheC._fields_}, "rec_k": MIS})
    assert lib.replayssm_gdn_decode(ctypes.byref(d), ctypes.byref(c2), FAKE, FAKE, FAKE, FAKE,
                                    FAKE, FAKE, None) == 2
    assert lib.replayssm_gdn_conventional_decode(ctypes.byref(d), None, FAKE, FAKE, FAKE, FAKE,
                                                 FAKE, FAKE, None) == 1
    d4 = rs.GDNDims(2, 4, 64, 64, 4)
    for T in (0, 5, 9):                          # draft counts outside 1..min(L, 8)
        assert lib.replayssm_gdn_verify(ctypes.byref(d4), ctypes.byref(c), T, FAKE, FAKE, FAKE, FAKE,
                                        FAKE, FAKE, None) == 4
        assert lib.replayssm_gdn_rollback(ctypes.byref(d4), ctypes.byref(c), T, FAKE, None) == 4
    assert lib.replayssm_gdn_verify(ctypes.byref(d4), ctypes.byref(c2), 2, FAKE, FAKE, FAKE, FAKE,
                                    FAKE, FAKE, None) == 2
    assert lib.replayssm_gdn_rollback(ctypes.byref(d4), ctypes.byref(c), 2, None, None) == 1


def test_capacity_checks(rs):
    """Cache capacity: negative, or below the batch without a slot map, is a
    shape error for both caches, before anything is launched; with a slot map any
    positive capacity passes the host checks."""
    lib = rs._lib
    d = _m2(rs, batch=4)
    assert _decode(rs, d, _cache(rs, capacity=-1)) == 3
    assert _decode(rs, d, _cache(rs, slots=None, capacity=3)) == 3
    assert lib.replayssm_rollback(ctypes.byref(d), ctypes.byref(_cache(rs, slots=None, capacity=2)), 1,
                                  FAKE, None) == 3
    assert lib.replayssm_flush(ctypes.byref(d), ctypes.byref(_cache(rs, capacity=-5)), None, None) == 3
    g = rs.GDNDims(4, 4, 64, 64, 16)
    base = {f: FAKE for f, _ in rs.GDNCacheC._fields_}
    for kw in ({"capacity": -1}, {"slots": None, "capacity": 3}):
        c = rs.GDNCacheC(**{**base, **kw})
        assert lib.replayssm_gdn_decode(ctypes.byref(g), ctypes.byref(c), FAKE, FAKE, FAKE, FAKE,
                                        FAKE, FAKE, None) == 3
        assert lib.replayssm_gdn_rollback(ctypes.byref(g), ctypes.byref(c), 1, FAKE, None) == 3


def test_noalloc_checks_before_anything(rs):
    """replayssm_decode_noalloc runs every host-side check of replayssm_decode
    (with cache->arrive allowed to be NULL: it supplies the counters itself) and
    its own capacity limit before it looks up or clears its counter array, so a
    rejected call enqueues nothing."""
    lib = rs._lib

    def na(dims, cache, dt=FAKE, x=FAKE):
        return lib.replayssm_decode_noalloc(ctypes.byref(dims), ctypes.byref(cache), dt, x, FAKE, FAKE,
                                            FAKE, None)

    assert lib.replayssm_decode_noalloc(None, ctypes.byref(_cache(rs)), FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert na(_m2(rs), _cache(rs, arrive=None), dt=None) == 1
    assert na(_m2(rs), _cache(rs, arrive=None, ckpt=None)) == 1
    assert na(_m2(rs), _cache(rs, arrive=None), x=MIS) == 2
    assert na(_m2(rs, dstate=48), _cache(rs, arrive=None)) == 3
    # the counter array holds 4096 sequences: a small batch through a slot map into
    # a larger cache is over the limit, and so is a batch of 4097 without a map
    assert na(_m2(rs, batch=4), _cache(rs, arrive=None, capacity=5000)) == 3
    assert na(_m2(rs, batch=4097), _cache(rs, arrive=None, slots=None, capacity=0)) == 3
