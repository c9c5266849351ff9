"""Gated DeltaNet speculative verify and rollback against the oracle.

Draft outputs against the stepwise oracle's verify (the FP32 gate), ring
pointers against the integer ring model, bit for bit; the drafts' records in
their ring slots, bit for bit; the checkpoint after a pre-flush against the
oracle state before the drafts.
"""
import numpy as np
import pytest
import torch

from oracle.gdn import GDNStepwise
from oracle.ring import RingModel
from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL, assert_close, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


class GDNVerifyRun:
    def __init__(self, shape, seed, T, sample=None):
        from ssm_decode_state_gb300 import replayssm as rs
        self.rs, self.shape, self.seed, self.T = rs, shape, seed, T
        b = shape.batch
        self.sample = np.arange(b) if sample is None else np.asarray(sample)
        S0 = gen.gdn_random_state(shape, seed)
        self.dims = rs.gdn_dims(b, shape.nheads, shape.dk, shape.dv, shape.L)
        self.cache = rs.gdn_cache(self.dims, ckpt=to_dev(S0))
        self.oracle = GDNStepwise(S0[self.sample])
        self.ring = RingModel(b, shape.L)
        self.records = {}                                  # tag -> (k, v, alpha, beta) of one sequence

    def _dev(self, st):
        return tuple(to_dev(a, torch.bfloat16) for a in (st.q, st.k, st.v)) + (to_dev(st.alpha), to_dev(st.beta))

    def decode(self, step):
        st = gen.gdn_step_inputs(self.shape, self.seed, 10_000 + step)
        o = self.rs.gdn_decode(self.cache, *self._dev(st))
        s = self.sample
        oo = self.oracle.step(st.q[s], st.k[s], st.v[s], st.alpha[s], st.beta[s])
        assert_close(o.cpu().numpy()[s], oo, f"gdn decode o step {step}", RTOL)
        self.ring.decode([("d", step)] * self.shape.batch)
        for b in s:
            self.records[(b, ("d", step))] = (st.k[b], st.v[b], st.alpha[b], st.beta[b])
        self.check_ring()

    def verify(self, step, accepted):
        T, s = self.T, self.sample
        st = gen.gdn_draft_inputs(self.shape, self.seed, step, T)
        before = self.oracle.S.copy()
        pre = np.asarray(self.ring.lens()) + T > self.shape.L
        o = self.rs.gdn_verify(self.cache, *self._dev(st))
        oo, states = self.oracle.verify(st.q[s], st.k[s], st.v[s], st.alpha[s], st.beta[s])
        assert_close(o.cpu().numpy()[s], oo, f"gdn verify o step {step}", RTOL)
        self.ring.verify([[("v", step, i) for i in range(T)] for _ in range(self.shape.batch)])
        for b in s:
            for i in range(T):
                self.records[(b, ("v", step, i))] = (st.k[b, i], st.v[b, i], st.alpha[b, i], st.beta[b, i])
        self.check_ring()
        self.check_records()
        for n, b in enumerate(s):
            if pre[b]:
                e = rel_err(self.cache.ckpt[b].cpu().numpy(), before[n])
                assert e <= RTOL, f"pre-flushed checkpoint of seq {b}, step {step}: {e:.3e}"
        acc = np.asarray(accepted, np.int32)
        self.rs.gdn_rollback(self.cache, T, torch.from_numpy(acc).cuda())
        self.oracle.accept(states, acc[s])
        self.ring.rollback(T, acc)
        self.check_ring()
        assert int(self.cache.err.item()) == 0
        return o, oo

    def check_ring(self):
        np.testing.assert_array_equal(self.cache.ring_len.cpu().numpy(), self.ring.lens())
        np.testing.assert_array_equal(self.cache.ring_head.cpu().numpy(), self.ring.heads())

    def check_records(self):
        rk = self.cache.rec_k.cpu().float().numpy()
        rv = self.cache.rec_v.cpu().float().numpy()
        ra = self.cache.rec_alpha.cpu().numpy()
        rb = self.cache.rec_beta.cpu().numpy()
        for b in self.sample:
            for slot, tag in self.ring.seqs[b].slots().items():
                k, v, al, be = self.records[(b, tag)]
                np.testing.assert_array_equal(rk[b, :, slot], _bf16(k))
                np.testing.assert_array_equal(rv[b, :, slot], _bf16(v))
                np.testing.assert_array_equal(ra[b, :, slot], al)
                np.testing.assert_array_equal(rb[b, :, slot], be)


@pytest.mark.parametrize("dk,dv,L,T", [(16, 16, 4, 2), (32, 24, 8, 3), (64, 64, 16, 4), (32, 32, 4, 4),
                                       (128, 128, 16, 4)])
def test_gdn_verify_rollback_small(dk, dv, L, T):
    """Verify + rollback over 3L steps (pre-flushes included), accepted counts
    drawn on 0..T, against the oracle and the ring model."""
    shape = gen.GDNShape(batch=5, nheads=3, dk=dk, dv=dv, L=L)
    r = GDNVerifyRun(shape, 700 + dk + T, T)
    for t in range(3 * L):
        r.verify(t, gen.accepted_counts(shape.batch, T, 700 + T, t))


def test_gdn_verify_one_draft_is_decode():
    """One draft scored by verify gives the decode output bit for bit (same
    chain, contraction and record-term order)."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.GDNShape(batch=3, nheads=4, dk=32, dv=32, L=8)
    S0 = gen.gdn_random_state(shape, 41)
    dims = rs.gdn_dims(3, 4, 32, 32, 8)
    c1 = rs.gdn_cache(dims, ckpt=to_dev(S0))
    c2 = rs.gdn_cache(dims, ckpt=to_dev(S0))
    for t in range(7):                                   # the ring never folds: decode and verify agree
        st = gen.gdn_step_inputs(shape, 41, t)
        args = tuple(to_dev(a, torch.bfloat16) for a in (st.q, st.k, st.v)) + (to_dev(st.alpha), to_dev(st.beta))
        o1 = rs.gdn_decode(c1, *args)
        o2 = rs.gdn_verify(c2, *(a[:, None] for a in args))[:, 0]
        np.testing.assert_array_equal(o1.cpu().numpy(), o2.cpu().numpy())
        np.testing.assert_array_equal(c1.ring_len.cpu().numpy(), c2.ring_len.cpu().numpy())


def test_gdn_decode_and_verify_mixed():
    """Decodes (folding on their own schedule) interleaved with verifies and
    rollbacks on the same cache."""
    shape = gen.GDNShape(batch=4, nheads=2, dk=64, dv=32, L=8)
    r = GDNVerifyRun(shape, 55, 3)
    rng = np.random.default_rng(2)
    for t in range(24):
        if t % 3 == 2:
            r.verify(t, rng.integers(0, 4, size=shape.batch).astype(np.int32))
        else:
            r.decode(t)


def test_gdn_verify_b256_T4_sampled():
    """Gated DeltaNet layer, batch 256, 32 heads, dk = dv = 128, L = 16: verify of
    4 drafts + rollback for 40 steps; the oracle follows 3 sequences."""
    w = gen.workloads()["gdn_verify_b256_T4"]
    r = GDNVerifyRun(w.shape, w.seed, w.T, sample=[0, 131, 255])
    for t in range(40):
        r.verify(t, gen.accepted_counts(w.shape.batch, w.T, w.seed, t))


@pytest.mark.parametrize("T,L", [(1, 4), (2, 8), (3, 16), (4, 4), (4, 16)])
def test_gdn_persistent_verify_variants(T, L):
    """The persistent verify (serving head shape, 12 sequences x 32 heads: more
    items than twice the SMs): draft counts 1..4 and rings of 4..16 over 3 L
    steps (pre-flushes included), accepted counts on 0..T, against the oracle's
    causal scoring, the ring model and the draft records."""
    shape = gen.GDNShape(batch=12, nheads=32, dk=128, dv=128, L=L)
    r = GDNVerifyRun(shape, 900 + 10 * T + L, T, sample=[0, 5, 11])
    for t in range(3 * L):
        r.verify(t, gen.accepted_counts(shape.batch, T, 900 + T, t))


def test_gdn_persistent_mixed_decode_verify():
    """Persistent decodes (folding on their own schedule) and persistent verifies
    with rollbacks interleaved on the same cache."""
    shape = gen.GDNShape(batch=12, nheads=32, dk=128, dv=128, L=8)
    r = GDNVerifyRun(shape, 57, 3, sample=[1, 10])
    rng = np.random.default_rng(4)
    for t in range(20):
        if t % 3 == 2:
            r.verify(t, rng.integers(0, 4, size=shape.batch).astype(np.int32))
        else:
            r.decode(t)


def test_gdn_persistent_decode_after_verify_fills_the_ring():
    """A verify that leaves exactly L records (L = 16, no pre-flush) followed by a
    persistent decode: the decode folds L + 1 records (the buffered ones and its
    token); outputs and the later steps stay on the oracle."""
    shape = gen.GDNShape(batch=12, nheads=32, dk=128, dv=128, L=16)
    r = GDNVerifyRun(shape, 211, 4, sample=[0, 7, 11])
    for t in range(12):                                  # 12 buffered records
        r.decode(t)
    r.verify(100, np.full(shape.batch, 4, np.int32))     # 12 + 4 = 16: no pre-flush, all accepted
    assert r.cache.ring_len.cpu().tolist() == [16] * shape.batch
    for t in range(12, 20):                              # the first of these folds 17 records
        r.decode(t)
    assert r.cache.ring_len.cpu().tolist() == [7] * shape.batch


def test_gdn_persistent_verify_bad_ring_pointers():
    """A sequence with invalid ring pointers is flagged and left untouched by the
    persistent verify; the other sequences proceed."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.GDNShape(batch=12, nheads=32, dk=128, dv=128, L=8)
    r = GDNVerifyRun(shape, 93, 2, sample=[0])
    r.verify(0, np.full(shape.batch, 2, np.int32))
    r.cache.ring_len[4] = 9                               # > L
    before = r.cache.ckpt[4].clone()
    rk = r.cache.rec_k[4].clone()
    d = gen.gdn_draft_inputs(shape, 93, 1, 2)
    rs.gdn_verify(r.cache, *r._dev(d))
    torch.cuda.synchronize()
    assert int(r.cache.err.item()) & rs.DEVERR_RING_META
    assert r.cache.ring_len[4].item() == 9 and r.cache.ring_len[0].item() == 4
    assert torch.equal(r.cache.ckpt[4], before) and torch.equal(r.cache.rec_k[4], rk)
    assert not r.cache.arrive.any().item()


def test_gdn_rollback_out_of_range():
    """An accepted count above T, or a ring too short to give back T - accepted
    records, leaves the sequence as it is and sets the rollback error bit."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.GDNShape(batch=3, nheads=2, dk=16, dv=16, L=8)
    r = GDNVerifyRun(shape, 9, 3)
    r.verify(0, np.array([3, 3, 3], np.int32))
    rs.gdn_rollback(r.cache, 3, torch.tensor([4, 1, -1], dtype=torch.int32, device="cuda"))
    assert r.cache.ring_len.cpu().tolist() == [3, 1, 3]
    assert int(r.cache.err.item()) == rs.DEVERR_ROLLBACK
