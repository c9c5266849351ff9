"""Cache-slot indirection (engine-style state indices for continuous batching).

A cache of `capacity` sequences driven through a map of distinct slots must do
exactly what a compacted cache (batch row b in slot b) holding the same
sequences does: the same outputs, bit for bit, the same state and records in
the mapped slots, and the unmapped slots untouched.  Exercised on the per-tile
and the persistent decode and verify, rollback, flush and the FP8 read copy.
"""
import numpy as np
import pytest
import torch

from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu

FIELDS = ("ckpt", "ckpt_q", "ckpt_scale", "rec_dt", "rec_x", "rec_B", "rec_C", "ring_head", "ring_len")


def _pair(shape, capacity, seed, read_copy=0):
    """A capacity-sized cache with random states in every slot, a random map of
    `batch` distinct slots, and the compacted cache of the mapped sequences."""
    from ssm_decode_state_gb300 import replayssm as rs
    prm = gen.mamba2_params(shape, seed)
    A, D = torch.from_numpy(prm.A), torch.from_numpy(prm.D)
    big_shape = gen.Mamba2Shape(capacity, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    h0 = to_dev(gen.mamba2_random_state(big_shape, seed))
    dims = rs.mamba2_dims(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L,
                          read_copy=read_copy)
    big = rs.mamba2_cache(dims, A, D, ckpt=h0.clone(), capacity=capacity)
    rng = np.random.default_rng(seed)
    slots = np.sort(rng.choice(capacity, size=shape.batch, replace=False)).astype(np.int32)
    rng.shuffle(slots)
    small = rs.mamba2_cache(dims, A, D, ckpt=h0[torch.from_numpy(slots).long()].clone())
    big.slots = torch.from_numpy(slots).cuda()
    if read_copy:
        rs.requant(big)
        rs.requant(small)
    return rs, prm, big, small, slots


def _check_same(big, small, slots, untouched=None):
    idx = torch.from_numpy(slots).long().cuda()
    for f in FIELDS:
        a, b = getattr(big, f), getattr(small, f)
        if a is None:
            continue
        assert torch.equal(a[idx], b), f
    if untouched is not None:
        for f, before in untouched.items():
            mask = torch.ones(getattr(big, f).shape[0], dtype=torch.bool, device="cuda")
            mask[idx] = False
            assert torch.equal(getattr(big, f)[mask], before[mask]), f"unmapped slots of {f} changed"
    assert int(big.err.item()) == 0 and int(small.err.item()) == 0


def _snapshot(cache):
    return {f: getattr(cache, f).clone() for f in FIELDS if getattr(cache, f) is not None}


def _dev_step(st):
    return (to_dev(st.dt), to_dev(st.x, torch.bfloat16), to_dev(st.B, torch.bfloat16), to_dev(st.C, torch.bfloat16))


@pytest.mark.parametrize("shape,capacity", [
    (gen.Mamba2Shape(batch=3, nheads=8, headdim=32, dstate=64, ngroups=2, L=4), 7),          # per-tile kernel
    (gen.Mamba2Shape(batch=48, nheads=128, headdim=64, dstate=128, ngroups=8, L=4), 80),     # persistent kernel
], ids=["per_tile", "persistent"])
def test_decode_through_slot_map(shape, capacity):
    rs, prm, big, small, slots = _pair(shape, capacity, 300 + capacity)
    before = _snapshot(big)
    for t in range(2 * shape.L + 1):                       # two folds per sequence
        args = _dev_step(gen.mamba2_step_inputs(shape, prm, 300, t))
        y1 = rs.decode(big, *args)
        y2 = rs.decode(small, *args)
        assert torch.equal(y1, y2), f"y differs at step {t}"
    _check_same(big, small, slots, untouched=before)


def test_decode_fp8_copy_through_slot_map():
    """The FP8 read path: codes and scales live in the mapped slots too."""
    shape = gen.Mamba2Shape(batch=32, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    rs, prm, big, small, slots = _pair(shape, 40, 91, read_copy=1)
    for t in range(2 * shape.L + 1):
        args = _dev_step(gen.mamba2_step_inputs(shape, prm, 91, t))
        assert torch.equal(rs.decode(big, *args), rs.decode(small, *args)), f"y differs at step {t}"
    _check_same(big, small, slots)


@pytest.mark.parametrize("shape,capacity,T", [
    (gen.Mamba2Shape(batch=4, nheads=8, headdim=32, dstate=64, ngroups=2, L=8), 9, 3),        # per-tile verify
    (gen.Mamba2Shape(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=8), 150, 4),  # persistent verify
], ids=["per_tile", "persistent"])
def test_verify_rollback_flush_through_slot_map(shape, capacity, T):
    rs, prm, big, small, slots = _pair(shape, capacity, 500 + T)
    before = _snapshot(big)
    for t in range(10):
        d = gen.mamba2_draft_inputs(shape, prm, 500, t, T)
        args = _dev_step(d)
        y1 = rs.verify(big, *args)
        y2 = rs.verify(small, *args)
        assert torch.equal(y1, y2), f"verify y differs at step {t}"
        acc = torch.from_numpy(gen.accepted_counts(shape.batch, T, 500, t)).cuda()
        rs.rollback(big, T, acc)
        rs.rollback(small, T, acc)
        if t % 4 == 3:                                     # a masked standalone flush now and then
            mask = torch.from_numpy((np.arange(shape.batch) % 2).astype(np.uint8)).cuda()
            rs.flush(big, mask)
            rs.flush(small, mask)
        _check_same(big, small, slots)
    _check_same(big, small, slots, untouched=before)


def test_slot_out_of_range_is_flagged_and_skipped():
    """A map entry outside [0, capacity) skips that row (nothing of the cache
    changes for it) and sets the slot error bit; the other rows proceed."""
    shape = gen.Mamba2Shape(batch=32, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    rs, prm, big, small, slots = _pair(shape, 40, 17)
    bad = slots.copy()
    bad[5] = 40                                            # == capacity
    before = _snapshot(big)
    args = _dev_step(gen.mamba2_step_inputs(shape, prm, 17, 0))
    rs.decode(big, *args, slots=torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert int(big.err.item()) & rs.DEVERR_SLOT
    s5 = int(slots[5])
    assert big.ring_len[s5].item() == 0 and torch.equal(big.ckpt[s5], before["ckpt"][s5])
    assert big.ring_len[int(slots[0])].item() == 1
    assert not big.arrive.any().item()


def test_decode_noalloc_through_slot_map():
    """The no-allocation entry keeps its arrival counters in library memory,
    sized by the capacity; through a slot map it matches the compacted cache."""
    shape = gen.Mamba2Shape(batch=64, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    rs, prm, big, small, slots = _pair(shape, 96, 23)
    before = _snapshot(big)
    for t in range(2 * shape.L + 1):
        args = _dev_step(gen.mamba2_step_inputs(shape, prm, 23, t))
        assert torch.equal(rs.decode_noalloc(big, *args), rs.decode(small, *args)), f"y differs at step {t}"
    _check_same(big, small, slots, untouched=before)


def test_duplicate_free_map_serves_a_changing_batch():
    """Continuous batching: sequences leave and join between steps; each step
    maps the live sequences to their slots, and every sequence ends where a
    private cache stepping only on its own live steps ends."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.Mamba2Shape(batch=4, nheads=8, headdim=32, dstate=64, ngroups=2, L=4)
    cap = 6
    prm = gen.mamba2_params(shape, 61)
    A, D = torch.from_numpy(prm.A), torch.from_numpy(prm.D)
    h0 = to_dev(gen.mamba2_random_state(gen.Mamba2Shape(cap, 8, 32, 64, 2, 4), 61))
    dims = rs.mamba2_dims(4, 8, 32, 64, 2, 4)
    big = rs.mamba2_cache(dims, A, D, ckpt=h0.clone(), capacity=cap)
    one = rs.mamba2_dims(1, 8, 32, 64, 2, 4)
    own = [rs.mamba2_cache(one, A, D, ckpt=h0[s:s + 1].clone()) for s in range(cap)]
    rng = np.random.default_rng(5)
    for t in range(13):
        live = rng.choice(cap, size=4, replace=False).astype(np.int32)
        args = _dev_step(gen.mamba2_step_inputs(shape, prm, 61, t))
        y = rs.decode(big, *args, slots=torch.from_numpy(live).cuda())
        for b, s in enumerate(live):
            ys = rs.decode(own[s], *(a[b:b + 1] for a in args))
            assert torch.equal(y[b:b + 1], ys), f"step {t}, row {b}, slot {s}"
    for s in range(cap):
        for f in FIELDS:
            a = getattr(big, f)
            if a is not None:
                assert torch.equal(a[s:s + 1], getattr(own[s], f)), f"slot {s} {f}"
    assert int(big.err.item()) == 0


# ------------------------------------------------------------------ Gated DeltaNet

GDN_FIELDS = ("ckpt", "rec_k", "rec_v", "rec_alpha", "rec_beta", "ring_head", "ring_len")


def _gdn_pair(shape, capacity, seed):
    from ssm_decode_state_gb300 import replayssm as rs
    big_shape = gen.GDNShape(capacity, shape.nheads, shape.dk, shape.dv, shape.L)
    S0 = to_dev(gen.gdn_random_state(big_shape, seed))
    dims = rs.gdn_dims(shape.batch, shape.nheads, shape.dk, shape.dv, shape.L)
    big = rs.gdn_cache(dims, ckpt=S0.clone(), capacity=capacity)
    rng = np.random.default_rng(seed)
    slots = rng.choice(capacity, size=shape.batch, replace=False).astype(np.int32)
    small = rs.gdn_cache(dims, ckpt=S0[torch.from_numpy(slots).long()].clone())
    big.slots = torch.from_numpy(slots).cuda()
    return rs, big, small, slots


def _gdn_check(big, small, slots, before=None):
    idx = torch.from_numpy(slots).long().cuda()
    for f in GDN_FIELDS:
        assert torch.equal(getattr(big, f)[idx], getattr(small, f)), f
    if before is not None:
        for f, b0 in before.items():
            mask = torch.ones(getattr(big, f).shape[0], dtype=torch.bool, device="cuda")
            mask[idx] = False
            assert torch.equal(getattr(big, f)[mask], b0[mask]), f"unmapped slots of {f} changed"
    assert int(big.err.item()) == 0 and int(small.err.item()) == 0


def _gdn_dev(st):
    return tuple(to_dev(a, torch.bfloat16) for a in (st.q, st.k, st.v)) + (to_dev(st.alpha), to_dev(st.beta))


@pytest.mark.parametrize("shape,capacity", [
    (gen.GDNShape(batch=24, nheads=32, dk=128, dv=128, L=4), 40),     # persistent decode
    (gen.GDNShape(batch=3, nheads=4, dk=64, dv=32, L=4), 7),          # per-tile decode
], ids=["persistent", "per_tile"])
def test_gdn_decode_through_slot_map(shape, capacity):
    rs, big, small, slots = _gdn_pair(shape, capacity, 400 + capacity)
    before = {f: getattr(big, f).clone() for f in GDN_FIELDS}
    for t in range(2 * shape.L + 1):
        args = _gdn_dev(gen.gdn_step_inputs(shape, 400, t))
        assert torch.equal(rs.gdn_decode(big, *args), rs.gdn_decode(small, *args)), f"o differs at step {t}"
    _gdn_check(big, small, slots, before)


def test_gdn_verify_rollback_flush_through_slot_map():
    shape = gen.GDNShape(batch=4, nheads=4, dk=64, dv=64, L=8)
    rs, big, small, slots = _gdn_pair(shape, 9, 41)
    before = {f: getattr(big, f).clone() for f in GDN_FIELDS}
    T = 3
    for t in range(8):
        args = _gdn_dev(gen.gdn_draft_inputs(shape, 41, t, T))
        assert torch.equal(rs.gdn_verify(big, *args), rs.gdn_verify(small, *args)), f"verify o differs at {t}"
        acc = torch.from_numpy(gen.accepted_counts(shape.batch, T, 41, t)).cuda()
        rs.gdn_rollback(big, T, acc)
        rs.gdn_rollback(small, T, acc)
        if t % 3 == 2:
            mask = torch.tensor([1, 0, 1, 1], dtype=torch.uint8, device="cuda")
            rs.gdn_flush(big, mask)
            rs.gdn_flush(small, mask)
        _gdn_check(big, small, slots)
    _gdn_check(big, small, slots, before)


def test_gdn_slot_out_of_range_is_flagged_and_skipped():
    shape = gen.GDNShape(batch=24, nheads=32, dk=128, dv=128, L=4)
    rs, big, small, slots = _gdn_pair(shape, 30, 43)
    bad = slots.copy()
    bad[3] = -1
    s3 = int(slots[3])
    ck3 = big.ckpt[s3].clone()
    rs.gdn_decode(big, *_gdn_dev(gen.gdn_step_inputs(shape, 43, 0)), slots=torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert int(big.err.item()) & rs.DEVERR_SLOT
    assert big.ring_len[s3].item() == 0 and torch.equal(big.ckpt[s3], ck3)
    assert big.ring_len[int(slots[0])].item() == 1
    assert not big.arrive.any().item()
