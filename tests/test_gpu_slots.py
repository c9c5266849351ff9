"""Cache-slot indirection (engine-style state indices for continuous batching).

A cache of `capacity` sequences driven through a map of distinct slots must do
exactly what a compacted cache (batch row b in slot b) holding the same
sequences does: the same outputs, bit for bit, the same state and records in
the mapped slots, and the unmapped slots untouched.  Exercised on the per-tile
and the persistent decode and verify, rollback, flush and the FP8 read copy.

Every test also follows cache slots with the oracle: the stepwise recurrence
of the sequence each slot holds and the integer ring model of its records.
Outputs of the rows mapped to a followed slot are checked against the oracle,
the ring pointers of the followed slots bit for bit against the ring model,
and their checkpoints after folds against the oracle's state.  A slot that
is not live on a step gets an identity token in the oracle (dt = 0 for
Mamba-2; alpha = 1, beta = 0 for Gated DeltaNet), which leaves its state
exactly as it is.
"""
import numpy as np
import pytest
import torch

from oracle.gdn import GDNStepwise
from oracle.mamba2 import Mamba2Stepwise
from oracle.ring import RingModel
from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL, assert_close, rel_err, to_dev

pytestmark = pytest.mark.gpu

FIELDS = ("ckpt", "ckpt_q", "ckpt_scale", "rec_dt", "rec_x", "rec_B", "rec_C", "ring_head", "ring_len")


class _M2Follow:
    """Oracle state and ring model of chosen cache slots of a Mamba-2 cache."""

    def __init__(self, prm, shape, h0_cap, slots):
        self.slots = [int(v) for v in slots]
        self.shape = shape
        self.orc = Mamba2Stepwise(prm.A, prm.D, shape.ngroups, h0_cap[self.slots])
        self.ring = RingModel(len(self.slots), shape.L)

    def _gather(self, st, row_of):
        """Inputs of the followed slots (identity token where a slot is not live)."""
        n = len(self.slots)
        dt = np.zeros((n,) + st.dt.shape[1:], np.float32)
        x = np.zeros((n,) + st.x.shape[1:], np.float32)
        B = np.zeros((n,) + st.B.shape[1:], np.float32)
        C = np.zeros((n,) + st.C.shape[1:], np.float32)
        live = np.zeros(n, bool)
        for i, sl in enumerate(self.slots):
            if sl in row_of:
                r = row_of[sl]
                dt[i], x[i], B[i], C[i], live[i] = st.dt[r], st.x[r], st.B[r], st.C[r], True
        return dt, x, B, C, live

    def decode(self, step, st, row_of, y, cache):
        """One decode token for the live followed slots; checks y of their rows,
        their ring pointers and, where they folded, their checkpoints."""
        dt, x, B, C, live = self._gather(st, row_of)
        yo = self.orc.step(dt, x, B, C)
        folded = [s.decode(step) if lv else None for s, lv in zip(self.ring.seqs, live)]
        yg = y.cpu().numpy()
        idx = [i for i in range(len(self.slots)) if live[i]]
        if idx:
            assert_close(yg[[row_of[self.slots[i]] for i in idx]], yo[idx], f"y through the map, step {step}")
        self.check(cache, [i for i, f in enumerate(folded) if f is not None])

    def verify(self, step, d, row_of, y, accepted):
        dt, x, B, C, live = self._gather(d, row_of)
        assert live.all()
        yo, states = self.orc.verify(dt, x, B, C)
        rows = [row_of[sl] for sl in self.slots]
        assert_close(y.cpu().numpy()[rows], yo, f"verify y through the map, step {step}")
        T = d.dt.shape[1]
        self.ring.verify([[(step, i) for i in range(T)] for _ in self.slots])
        acc = np.asarray(accepted)[rows]
        self.orc.accept(states, acc)
        self.ring.rollback(T, acc)

    def flush(self, mask_of_slot, cache):
        m = [bool(mask_of_slot.get(sl, False)) for sl in self.slots]
        self.ring.flush(m)
        self.check(cache, [i for i, v in enumerate(m) if v])

    def check(self, cache, ckpt_idx=()):
        sl = torch.tensor(self.slots, dtype=torch.long, device="cuda")
        np.testing.assert_array_equal(cache.ring_head[sl].cpu().numpy(), self.ring.heads())
        np.testing.assert_array_equal(cache.ring_len[sl].cpu().numpy(), self.ring.lens())
        for i in ckpt_idx:
            e = rel_err(cache.ckpt[self.slots[i]].cpu().numpy(), self.orc.h[i])
            assert e <= RTOL, f"checkpoint of slot {self.slots[i]}: {e:.3e}"


def _pair(shape, capacity, seed, read_copy=0):
    """A capacity-sized cache with random states in every slot, a random map of
    `batch` distinct slots, and the compacted cache of the mapped sequences."""
    from ssm_decode_state_gb300 import replayssm as rs
    prm = gen.mamba2_params(shape, seed)
    A, D = torch.from_numpy(prm.A), torch.from_numpy(prm.D)
    big_shape = gen.Mamba2Shape(capacity, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    h0_host = gen.mamba2_random_state(big_shape, seed)
    h0 = to_dev(h0_host)
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
    return rs, prm, big, small, slots, h0_host


def _follow_rows(shape, prm, h0_host, slots, rows):
    """Oracle follower of the slots that batch rows `rows` map to."""
    return _M2Follow(prm, shape, h0_host, [slots[r] for r in rows])


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
    (gen.Mamba2Shape(batch=5, nheads=128, headdim=64, dstate=128, ngroups=8, L=4), 12),      # small-batch kernel
    (gen.Mamba2Shape(batch=1, nheads=128, headdim=64, dstate=128, ngroups=8, L=4), 9),       # small-batch kernel, batch 1
], ids=["per_tile", "persistent", "small_batch", "small_batch_1"])
def test_decode_through_slot_map(shape, capacity):
    rs, prm, big, small, slots, h0 = _pair(shape, capacity, 300 + capacity)
    rows = sorted({0, shape.batch // 2, shape.batch - 1})
    fol = _follow_rows(shape, prm, h0, slots, rows)
    row_of = {int(slots[r]): r for r in rows}
    del h0
    before = _snapshot(big)
    for t in range(2 * shape.L + 1):                       # two folds per sequence
        st = gen.mamba2_step_inputs(shape, prm, 300, t)
        args = _dev_step(st)
        y1 = rs.decode(big, *args)
        y2 = rs.decode(small, *args)
        assert torch.equal(y1, y2), f"y differs at step {t}"
        fol.decode(t, st, row_of, y1, big)
    _check_same(big, small, slots, untouched=before)


def test_decode_fp8_copy_through_slot_map():
    """The FP8 read path: codes and scales live in the mapped slots too."""
    shape = gen.Mamba2Shape(batch=32, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    rs, prm, big, small, slots, h0 = _pair(shape, 40, 91, read_copy=1)
    rows = [0, shape.batch - 1]
    fol = _follow_rows(shape, prm, h0, slots, rows)
    row_of = {int(slots[r]): r for r in rows}
    del h0
    for t in range(2 * shape.L + 1):
        st = gen.mamba2_step_inputs(shape, prm, 91, t)
        args = _dev_step(st)
        y = rs.decode(big, *args)
        assert torch.equal(y, rs.decode(small, *args)), f"y differs at step {t}"
        if (t + 1) % shape.L == 0:
            # fold step: y from the FP32 checkpoint, checked against the oracle with
            # the folded checkpoints
            fol.decode(t, st, row_of, y, big)
        else:
            # read-copy step: ring pointers against the ring model (the FP8 error
            # bound of y is checked by the read-copy tests)
            dt, x, B, C, _ = fol._gather(st, row_of)
            fol.orc.step(dt, x, B, C)
            for sq in fol.ring.seqs:
                sq.decode(t)
            fol.check(big)
    _check_same(big, small, slots)


@pytest.mark.parametrize("shape,capacity,T", [
    (gen.Mamba2Shape(batch=4, nheads=8, headdim=32, dstate=64, ngroups=2, L=8), 9, 3),        # per-tile verify
    (gen.Mamba2Shape(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=8), 150, 4),  # persistent verify
], ids=["per_tile", "persistent"])
def test_verify_rollback_flush_through_slot_map(shape, capacity, T):
    rs, prm, big, small, slots, h0 = _pair(shape, capacity, 500 + T)
    rows = sorted({0, 1, shape.batch // 2, shape.batch - 1})
    fol = _follow_rows(shape, prm, h0, slots, rows)
    row_of = {int(slots[r]): r for r in rows}
    del h0
    before = _snapshot(big)
    for t in range(10):
        d = gen.mamba2_draft_inputs(shape, prm, 500, t, T)
        args = _dev_step(d)
        y1 = rs.verify(big, *args)
        y2 = rs.verify(small, *args)
        assert torch.equal(y1, y2), f"verify y differs at step {t}"
        acc_np = gen.accepted_counts(shape.batch, T, 500, t)
        acc = torch.from_numpy(acc_np).cuda()
        rs.rollback(big, T, acc)
        rs.rollback(small, T, acc)
        fol.verify(t, d, row_of, y1, acc_np)
        fol.check(big)
        if t % 4 == 3:                                     # a masked standalone flush now and then
            mask_np = (np.arange(shape.batch) % 2).astype(np.uint8)
            mask = torch.from_numpy(mask_np).cuda()
            rs.flush(big, mask)
            rs.flush(small, mask)
            fol.flush({int(slots[r]): mask_np[r] for r in rows}, big)
        _check_same(big, small, slots)
    _check_same(big, small, slots, untouched=before)


@pytest.mark.parametrize("batch", [32, 8], ids=["persistent", "small_batch"])
def test_slot_out_of_range_is_flagged_and_skipped(batch):
    """A map entry outside [0, capacity) skips that row (nothing of the cache
    changes for it) and sets the slot error bit; the other rows proceed."""
    shape = gen.Mamba2Shape(batch=batch, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    rs, prm, big, small, slots, h0 = _pair(shape, 40, 17)
    last = batch - 1
    fol = _follow_rows(shape, prm, h0, slots, [0, last])
    del h0
    bad = slots.copy()
    bad[5] = 40                                            # == capacity
    before = _snapshot(big)
    st = gen.mamba2_step_inputs(shape, prm, 17, 0)
    args = _dev_step(st)
    y = rs.decode(big, *args, slots=torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert int(big.err.item()) & rs.DEVERR_SLOT
    big.err.zero_()
    fol.decode(0, st, {int(slots[0]): 0, int(slots[last]): last}, y, big)   # the other rows proceed
    s5 = int(slots[5])
    assert big.ring_len[s5].item() == 0 and torch.equal(big.ckpt[s5], before["ckpt"][s5])
    assert big.ring_len[int(slots[0])].item() == 1
    assert not big.arrive.any().item()


def test_decode_noalloc_through_slot_map():
    """The no-allocation entry keeps its arrival counters in library memory,
    sized by the capacity; through a slot map it matches the compacted cache."""
    shape = gen.Mamba2Shape(batch=64, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    rs, prm, big, small, slots, h0 = _pair(shape, 96, 23)
    rows = [0, 33, 63]
    fol = _follow_rows(shape, prm, h0, slots, rows)
    row_of = {int(slots[r]): r for r in rows}
    del h0
    before = _snapshot(big)
    for t in range(2 * shape.L + 1):
        st = gen.mamba2_step_inputs(shape, prm, 23, t)
        args = _dev_step(st)
        y = rs.decode_noalloc(big, *args)
        assert torch.equal(y, rs.decode(small, *args)), f"y differs at step {t}"
        fol.decode(t, st, row_of, y, big)
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
    fol = _M2Follow(prm, shape, h0.cpu().numpy(), range(cap))       # every slot
    rng = np.random.default_rng(5)
    for t in range(13):
        live = rng.choice(cap, size=4, replace=False).astype(np.int32)
        st = gen.mamba2_step_inputs(shape, prm, 61, t)
        args = _dev_step(st)
        y = rs.decode(big, *args, slots=torch.from_numpy(live).cuda())
        for b, s in enumerate(live):
            ys = rs.decode(own[s], *(a[b:b + 1] for a in args))
            assert torch.equal(y[b:b + 1], ys), f"step {t}, row {b}, slot {s}"
        fol.decode(t, st, {int(s): b for b, s in enumerate(live)}, y, big)
    for s in range(cap):
        for f in FIELDS:
            a = getattr(big, f)
            if a is not None:
                assert torch.equal(a[s:s + 1], getattr(own[s], f)), f"slot {s} {f}"
    assert int(big.err.item()) == 0


# ------------------------------------------------------------------ Gated DeltaNet

GDN_FIELDS = ("ckpt", "rec_k", "rec_v", "rec_alpha", "rec_beta", "ring_head", "ring_len")


class _GDNFollow:
    """Oracle state and ring model of chosen cache slots of a Gated DeltaNet cache."""

    def __init__(self, shape, S0_cap, slots):
        self.slots = [int(v) for v in slots]
        self.shape = shape
        self.orc = GDNStepwise(S0_cap[self.slots])
        self.ring = RingModel(len(self.slots), shape.L)

    def _gather(self, st, row_of):
        n = len(self.slots)
        q = np.zeros((n,) + st.q.shape[1:], np.float32)
        k = np.zeros((n,) + st.k.shape[1:], np.float32)
        v = np.zeros((n,) + st.v.shape[1:], np.float32)
        al = np.ones((n,) + st.alpha.shape[1:], np.float32)       # identity token: alpha 1, beta 0
        be = np.zeros((n,) + st.beta.shape[1:], np.float32)
        live = np.zeros(n, bool)
        for i, sl in enumerate(self.slots):
            if sl in row_of:
                r = row_of[sl]
                q[i], k[i], v[i], al[i], be[i], live[i] = st.q[r], st.k[r], st.v[r], st.alpha[r], st.beta[r], True
        return q, k, v, al, be, live

    def decode(self, step, st, row_of, o, cache):
        q, k, v, al, be, live = self._gather(st, row_of)
        oo = self.orc.step(q, k, v, al, be)
        folded = [s.decode(step) if lv else None for s, lv in zip(self.ring.seqs, live)]
        idx = [i for i in range(len(self.slots)) if live[i]]
        if idx:
            assert_close(o.cpu().numpy()[[row_of[self.slots[i]] for i in idx]], oo[idx],
                         f"gdn o through the map, step {step}")
        self.check(cache, [i for i, f in enumerate(folded) if f is not None])

    def verify(self, step, d, row_of, o, accepted):
        q, k, v, al, be, live = self._gather(d, row_of)
        assert live.all()
        oo, states = self.orc.verify(q, k, v, al, be)
        rows = [row_of[sl] for sl in self.slots]
        assert_close(o.cpu().numpy()[rows], oo, f"gdn verify o through the map, step {step}")
        T = d.alpha.shape[1]
        self.ring.verify([[(step, i) for i in range(T)] for _ in self.slots])
        acc = np.asarray(accepted)[rows]
        self.orc.accept(states, acc)
        self.ring.rollback(T, acc)

    def flush(self, mask_of_slot, cache):
        m = [bool(mask_of_slot.get(sl, False)) for sl in self.slots]
        self.ring.flush(m)
        self.check(cache, [i for i, v in enumerate(m) if v])

    def check(self, cache, ckpt_idx=()):
        sl = torch.tensor(self.slots, dtype=torch.long, device="cuda")
        np.testing.assert_array_equal(cache.ring_head[sl].cpu().numpy(), self.ring.heads())
        np.testing.assert_array_equal(cache.ring_len[sl].cpu().numpy(), self.ring.lens())
        for i in ckpt_idx:
            e = rel_err(cache.ckpt[self.slots[i]].cpu().numpy(), self.orc.S[i])
            assert e <= RTOL, f"checkpoint of slot {self.slots[i]}: {e:.3e}"


def _gdn_pair(shape, capacity, seed):
    from ssm_decode_state_gb300 import replayssm as rs
    big_shape = gen.GDNShape(capacity, shape.nheads, shape.dk, shape.dv, shape.L)
    S0_host = gen.gdn_random_state(big_shape, seed)
    S0 = to_dev(S0_host)
    dims = rs.gdn_dims(shape.batch, shape.nheads, shape.dk, shape.dv, shape.L)
    big = rs.gdn_cache(dims, ckpt=S0.clone(), capacity=capacity)
    rng = np.random.default_rng(seed)
    slots = rng.choice(capacity, size=shape.batch, replace=False).astype(np.int32)
    small = rs.gdn_cache(dims, ckpt=S0[torch.from_numpy(slots).long()].clone())
    big.slots = torch.from_numpy(slots).cuda()
    return rs, big, small, slots, S0_host


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
    rs, big, small, slots, S0 = _gdn_pair(shape, capacity, 400 + capacity)
    rows = sorted({0, shape.batch // 2, shape.batch - 1})
    fol = _GDNFollow(shape, S0, [slots[r] for r in rows])
    row_of = {int(slots[r]): r for r in rows}
    before = {f: getattr(big, f).clone() for f in GDN_FIELDS}
    for t in range(2 * shape.L + 1):
        st = gen.gdn_step_inputs(shape, 400, t)
        args = _gdn_dev(st)
        o = rs.gdn_decode(big, *args)
        assert torch.equal(o, rs.gdn_decode(small, *args)), f"o differs at step {t}"
        fol.decode(t, st, row_of, o, big)
    _gdn_check(big, small, slots, before)


@pytest.mark.parametrize("shape,capacity", [
    (gen.GDNShape(batch=4, nheads=4, dk=64, dv=64, L=8), 9),          # per-tile verify
    (gen.GDNShape(batch=16, nheads=32, dk=128, dv=128, L=8), 24),     # persistent verify
], ids=["per_tile", "persistent"])
def test_gdn_verify_rollback_flush_through_slot_map(shape, capacity):
    rs, big, small, slots, S0 = _gdn_pair(shape, capacity, 41)
    fol = _GDNFollow(shape, S0, slots)                     # every row
    row_of = {int(sl): r for r, sl in enumerate(slots)}
    before = {f: getattr(big, f).clone() for f in GDN_FIELDS}
    T = 3
    for t in range(8):
        d = gen.gdn_draft_inputs(shape, 41, t, T)
        args = _gdn_dev(d)
        o = rs.gdn_verify(big, *args)
        assert torch.equal(o, rs.gdn_verify(small, *args)), f"verify o differs at {t}"
        acc_np = gen.accepted_counts(shape.batch, T, 41, t)
        acc = torch.from_numpy(acc_np).cuda()
        rs.gdn_rollback(big, T, acc)
        rs.gdn_rollback(small, T, acc)
        fol.verify(t, d, row_of, o, acc_np)
        fol.check(big)
        if t % 3 == 2:
            mask_np = (np.arange(shape.batch) % 4 != 1).astype(np.uint8)
            mask = torch.from_numpy(mask_np).cuda()
            rs.gdn_flush(big, mask)
            rs.gdn_flush(small, mask)
            fol.flush({int(slots[r]): mask_np[r] for r in range(shape.batch)}, big)
        _gdn_check(big, small, slots)
    _gdn_check(big, small, slots, before)


def test_gdn_slot_out_of_range_is_flagged_and_skipped():
    shape = gen.GDNShape(batch=24, nheads=32, dk=128, dv=128, L=4)
    rs, big, small, slots, S0 = _gdn_pair(shape, 30, 43)
    fol = _GDNFollow(shape, S0, [slots[0], slots[23]])
    bad = slots.copy()
    bad[3] = -1
    s3 = int(slots[3])
    ck3 = big.ckpt[s3].clone()
    st = gen.gdn_step_inputs(shape, 43, 0)
    o = rs.gdn_decode(big, *_gdn_dev(st), slots=torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert int(big.err.item()) & rs.DEVERR_SLOT
    fol.decode(0, st, {int(slots[0]): 0, int(slots[23]): 23}, o, big)    # the other rows proceed
    assert big.ring_len[s3].item() == 0 and torch.equal(big.ckpt[s3], ck3)
    assert big.ring_len[int(slots[0])].item() == 1
    assert not big.arrive.any().item()


def test_gdn_changing_batch_against_oracle():
    """Continuous batching on the Gated DeltaNet cache (persistent kernel):
    live sequences change every step; every slot is followed by the oracle (idle
    slots take identity tokens), so outputs, ring pointers and folded
    checkpoints of every slot are checked as the live set changes."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.GDNShape(batch=12, nheads=32, dk=128, dv=128, L=4)
    cap = 20
    S0 = gen.gdn_random_state(gen.GDNShape(cap, 32, 128, 128, 4), 83)
    dims = rs.gdn_dims(shape.batch, 32, 128, 128, 4)
    big = rs.gdn_cache(dims, ckpt=to_dev(S0), capacity=cap)
    fol = _GDNFollow(shape, S0, range(cap))
    rng = np.random.default_rng(8)
    for t in range(14):
        live = rng.choice(cap, size=shape.batch, replace=False).astype(np.int32)
        st = gen.gdn_step_inputs(shape, 83, t)
        o = rs.gdn_decode(big, *_gdn_dev(st), slots=torch.from_numpy(live).cuda())
        fol.decode(t, st, {int(s_): b for b, s_ in enumerate(live)}, o, big)
    assert int(big.err.item()) == 0 and not big.arrive.any().item()
