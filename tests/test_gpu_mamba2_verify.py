"""Speculative verify, rollback, standalone flush and the snapshot-per-draft
comparison path, against the oracle and the integer ring model."""
import numpy as np
import pytest
import torch

from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL_INPLACE, assert_close, io_dtype, to_dev

pytestmark = pytest.mark.gpu


class VerifyRun:
    """Replay cache + snapshot pool on the GPU, oracle on `sample`."""

    def __init__(self, shape, seed, T, sample=None, h0=None, conventional=True):
        from ssm_decode_state_gb300 import replayssm as rs
        from tests.m2_runner import M2Run
        self.rs = rs
        self.r = M2Run(shape, seed, h0=h0, sample=sample, conventional=False)
        self.T = T
        self.shape = shape
        b = shape.batch
        if conventional:
            h0d = self.r.cache.ckpt.clone()
            self.pool = torch.zeros((b, T + 1) + tuple(h0d.shape[1:]), device="cuda")
            self.pool[:, 0] = h0d
            self.slot = torch.zeros(b, dtype=torch.int32, device="cuda")
            self.cerr = torch.zeros(1, dtype=torch.int32, device="cuda")
        else:
            self.pool = None

    def dev(self, st):
        io = io_dtype(self.shape.bf16_io)
        return to_dev(st.dt), to_dev(st.x, io), to_dev(st.B, io), to_dev(st.C, io)

    def verify_step(self, step, accepted, check=True):
        r, rs, T = self.r, self.rs, self.T
        d = gen.mamba2_draft_inputs(self.shape, r.params, self.r.seed, step, T)
        dt, x, B, C = self.dev(d)
        y = rs.verify(r.cache, dt, x, B, C)
        s = r.sample
        yo, states = r.oracle.verify(d.dt[s], d.x[s], d.B[s], d.C[s])
        r.ring.verify([[(step, i) for i in range(T)] for _ in range(self.shape.batch)])
        r._keep(step, d)
        if check:
            assert_close(y.cpu().numpy()[s], yo, f"verify y step {step}")
        if self.pool is not None:
            yc = rs.conventional_verify(r.dims, self.pool, self.slot, r.cache.A, r.cache.D, dt, x, B, C,
                                        self.cerr)
            if check:
                assert_close(yc.cpu().numpy()[s], yo, f"snapshot verify y step {step}", RTOL_INPLACE)
        acc = torch.from_numpy(accepted.astype(np.int32)).cuda()
        rs.rollback(r.cache, T, acc)
        if self.pool is not None:
            rs.conventional_select(self.slot, T, acc, self.cerr)
        r.oracle.accept(states, accepted[s])
        r.ring.rollback(T, accepted)
        if check:
            r.check_ring()
        return y, yo


def test_verify_T1_equals_decode():
    """One draft scored by verify gives the decode output, bit for bit."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.Mamba2Shape(batch=3, nheads=8, headdim=32, dstate=64, ngroups=2, L=8)
    h0 = gen.mamba2_random_state(shape, 31)
    prm = gen.mamba2_params(shape, 31)
    dims = rs.mamba2_dims(3, 8, 32, 64, 2, 8)
    A, D = torch.from_numpy(prm.A), torch.from_numpy(prm.D)
    c1 = rs.mamba2_cache(dims, A, D, ckpt=to_dev(h0))
    c2 = rs.mamba2_cache(dims, A, D, ckpt=to_dev(h0))
    for t in range(11):
        st = gen.mamba2_step_inputs(shape, prm, 31, t)
        dt, x, B, C = to_dev(st.dt), to_dev(st.x, torch.bfloat16), to_dev(st.B, torch.bfloat16), \
            to_dev(st.C, torch.bfloat16)
        y1 = rs.decode(c1, dt, x, B, C)
        y2 = rs.verify(c2, dt[:, None], x[:, None], B[:, None], C[:, None])[:, 0]
        np.testing.assert_array_equal(y1.cpu().numpy(), y2.cpu().numpy())
        # verify never folds its draft; where decode folded, flush the same records
        if int(c1.ring_len[0].item()) == 0:
            rs.flush(c2)
            np.testing.assert_array_equal(c1.ckpt.cpu().numpy(), c2.ckpt.cpu().numpy())


@pytest.mark.parametrize("T,L", [(4, 16), (3, 4), (1, 4), (8, 8)])
def test_verify_rollback_small(T, L):
    shape = gen.Mamba2Shape(batch=5, nheads=8, headdim=16, dstate=32, ngroups=2, L=L)
    h0 = gen.mamba2_random_state(shape, 40 + T)
    v = VerifyRun(shape, 40 + T, T, h0=h0)
    for t in range(24):
        acc = gen.accepted_counts(shape.batch, T, 40 + T, t)
        v.verify_step(t, acc)
        if t % 5 == 0:
            v.r.check_records()


def test_mixed_decode_verify_rollback():
    """Decode steps interleaved with verify/rollback, including a decode that
    meets a full ring (verify left exactly L records) and folds L + 1."""
    shape = gen.Mamba2Shape(batch=4, nheads=8, headdim=16, dstate=32, ngroups=2, L=4)
    h0 = gen.mamba2_random_state(shape, 55)
    v = VerifyRun(shape, 55, 2, h0=h0, conventional=False)
    r = v.r
    rng = np.random.default_rng(0)
    for t in range(40):
        if t % 3 == 2:
            acc = rng.integers(0, 3, size=shape.batch).astype(np.int32)
            acc[t % shape.batch] = 2
            v.verify_step(10_000 + t, acc)
        else:
            r.decode(20_000 + t)
        r.check_records()


def test_standalone_flush_masked():
    from ssm_decode_state_gb300 import replayssm as rs
    from tests.m2_runner import M2Run
    shape = gen.Mamba2Shape(batch=4, nheads=8, headdim=32, dstate=64, ngroups=2, L=16)
    h0 = gen.mamba2_random_state(shape, 66)
    r = M2Run(shape, 66, h0=h0)
    for t in range(5):
        r.decode(t)
    mask = torch.tensor([1, 0, 1, 0], dtype=torch.uint8, device="cuda")
    rs.flush(r.cache, mask)
    r.ring.flush([True, False, True, False])
    r.check_ring()
    r.check_ckpt(-1, seqs=[0, 2])
    ck = r.cache.ckpt.cpu().numpy()
    np.testing.assert_array_equal(ck[1], h0[1])          # untouched
    for t in range(5, 20):
        r.decode(t)
    rs.flush(r.cache)                                       # all, incl. empty rings
    r.ring.flush()
    r.check_ring()
    r.check_ckpt(-1)


def test_rollback_is_pointer_move_bitwise():
    """verify(T) + rollback(a) leaves exactly the state of a run that never saw
    the rejected drafts: the same flush decision (standalone flush where
    len + T > L), then verify of only the a accepted drafts.  Checkpoint, ring
    pointers and live records match bit for bit, and so do all later outputs."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.Mamba2Shape(batch=4, nheads=8, headdim=32, dstate=64, ngroups=2, L=8)
    T, seed = 4, 77
    prm = gen.mamba2_params(shape, seed)
    h0 = gen.mamba2_random_state(shape, seed)
    A, D = torch.from_numpy(prm.A), torch.from_numpy(prm.D)
    runA = rs.mamba2_cache(rs.mamba2_dims(4, 8, 32, 64, 2, 8), A, D, ckpt=to_dev(h0))
    dims1 = rs.mamba2_dims(1, 8, 32, 64, 2, 8)
    runB = [rs.mamba2_cache(dims1, A, D, ckpt=to_dev(h0[i:i + 1])) for i in range(4)]

    def dec(cache, st, sl=slice(None)):
        return rs.decode(cache, to_dev(st.dt[sl]), to_dev(st.x[sl], torch.bfloat16),
                         to_dev(st.B[sl], torch.bfloat16), to_dev(st.C[sl], torch.bfloat16))

    for t in range(5):                                      # len 5 everywhere
        st = gen.mamba2_step_inputs(shape, prm, seed, t)
        dec(runA, st)
        for i in range(4):
            dec(runB[i], st, slice(i, i + 1))
    for rnd in range(6):
        d = gen.mamba2_draft_inputs(shape, prm, seed, 100 + rnd, T)
        acc = np.array([0, 1, 3, 4], np.int32)[np.roll(np.arange(4), rnd)]
        lens = runA.ring_len.cpu().numpy()
        rs.verify(runA, to_dev(d.dt), to_dev(d.x, torch.bfloat16), to_dev(d.B, torch.bfloat16),
                  to_dev(d.C, torch.bfloat16))
        rs.rollback(runA, T, torch.from_numpy(acc).cuda())
        for i in range(4):
            if lens[i] + T > 8:
                rs.flush(runB[i])
            a = int(acc[i])
            if a:
                sl = slice(i, i + 1)
                rs.verify(runB[i], to_dev(d.dt[sl, :a]), to_dev(d.x[sl, :a], torch.bfloat16),
                          to_dev(d.B[sl, :a], torch.bfloat16), to_dev(d.C[sl, :a], torch.bfloat16))
        for i in range(4):
            np.testing.assert_array_equal(runA.ckpt[i].cpu().numpy(), runB[i].ckpt[0].cpu().numpy())
            assert runA.ring_head[i].item() == runB[i].ring_head[0].item()
            ln = runA.ring_len[i].item()
            assert ln == runB[i].ring_len[0].item()
            hd = runA.ring_head[i].item()
            for j in range(ln):
                sl = (hd + j) % 8
                for f in ("rec_dt", "rec_x", "rec_B", "rec_C"):
                    np.testing.assert_array_equal(getattr(runA, f)[i, :, sl].float().cpu().numpy(),
                                                  getattr(runB[i], f)[0, :, sl].float().cpu().numpy())
        st = gen.mamba2_step_inputs(shape, prm, seed, 1000 + rnd)
        yA = dec(runA, st).cpu().numpy()
        for i in range(4):
            np.testing.assert_array_equal(yA[i], dec(runB[i], st, slice(i, i + 1)).cpu().numpy()[0])


def test_verify_serving_shape_b512_sampled():
    """Speculative verify on the serving head shape at batch 512: T = 4 drafts
    per step, accepted prefix uniform on {0..4}, 200 steps; the oracle follows
    3 sequences, the snapshot-per-draft path is compared too, ring pointers of
    all 512 sequences bit-exact at every step."""
    w = gen.workloads()["mamba2_verify_b512_T4"]
    h0 = gen.mamba2_random_state(w.shape, w.seed)
    v = VerifyRun(w.shape, w.seed, w.T, sample=[0, 300, 511], h0=h0)
    del h0
    for t in range(w.steps):
        acc = gen.accepted_counts(w.shape.batch, w.T, w.seed, t)
        v.verify_step(t, acc)
    v.r.check_records(seqs=[0, 300, 511])


def test_snapshot_slot_bounds_and_select():
    from ssm_decode_state_gb300 import replayssm as rs
    slot = torch.tensor([0, 4, 2], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs.conventional_select(slot, 4, torch.tensor([3, 2, 4], dtype=torch.int32, device="cuda"), err)
    assert slot.cpu().tolist() == [3, 1, 1] and err.item() == 0
    rs.conventional_select(slot, 4, torch.tensor([5, 0, -1], dtype=torch.int32, device="cuda"), err)
    assert slot.cpu().tolist() == [3, 1, 1] and err.item() == rs.DEVERR_ROLLBACK


@pytest.mark.parametrize("T,L", [(1, 8), (3, 8), (4, 8), (4, 16), (4, 4)])
def test_persistent_verify_variants(T, L):
    """Serving head shape at batch 128 (the persistent verify): 1-4 drafts, rings
    of 8 (pre-flush every couple of steps) and 16; outputs against the oracle,
    ring pointers of all sequences and the live records bit-exact."""
    shape = gen.Mamba2Shape(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=L)
    h0 = gen.mamba2_random_state(shape, 500 + T)
    v = VerifyRun(shape, 500 + T, T, h0=h0, sample=[0, 77, 127], conventional=False)
    del h0
    for t in range(14):
        v.verify_step(t, gen.accepted_counts(shape.batch, T, 500 + T, t))
        if t % 4 == 3:
            v.r.check_records(seqs=[0, 77, 127])


def test_persistent_mixed_decode_verify():
    """Persistent decode and persistent verify on the same cache, interleaved,
    including decodes that meet a ring a verify left full."""
    shape = gen.Mamba2Shape(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=8)
    h0 = gen.mamba2_random_state(shape, 612)
    v = VerifyRun(shape, 612, 4, h0=h0, sample=[5, 120], conventional=False)
    del h0
    rng = np.random.default_rng(3)
    for t in range(30):
        if t % 3 == 1:
            acc = rng.integers(0, 5, size=shape.batch).astype(np.int32)
            acc[::7] = 4
            v.verify_step(40_000 + t, acc)
        else:
            v.r.decode(50_000 + t)
        if t % 5 == 0:
            v.r.check_records(seqs=[5, 120])


def test_persistent_verify_fp8_copy_preflush():
    """With an FP8 read copy, a pre-flushing verify rebuilds the copy of the new
    checkpoint (every code within half an E4M3 step of the FP32 value)."""
    from tests.m2_runner import M2Run
    shape = gen.Mamba2Shape(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    h0 = gen.mamba2_random_state(shape, 71)
    r = M2Run(shape, 71, h0=h0, read_copy=1, sample=[9], conventional=False)
    del h0
    v = VerifyRun.__new__(VerifyRun)
    from ssm_decode_state_gb300 import replayssm as rs
    v.rs, v.r, v.T, v.shape, v.pool = rs, r, 3, shape, None
    for t in range(4):
        v.verify_step(t, gen.accepted_counts(shape.batch, 3, 71, t))
    ck = r.cache.ckpt[:8].cpu().numpy().astype(np.float64)
    sc = r.cache.ckpt_scale[:8].cpu().numpy().astype(np.float64)
    codes = r.cache.ckpt_q[:8].cpu().numpy()
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e, m = (codes >> 3) & 0xF, codes & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7))
    dq = sign * mag * sc[..., None]
    assert np.all(np.abs(dq - ck) <= 2.0 ** -4 * np.abs(ck) + 2.0 ** -10 * sc[..., None] + 1e-6 * np.abs(ck))


def test_persistent_verify_bad_ring_pointers():
    """Serving head shape at batch 128 (the persistent verify): a sequence with
    invalid ring pointers is flagged and left untouched (checkpoint, records,
    pointers); the other sequences take their drafts."""
    from ssm_decode_state_gb300 import replayssm as rs
    from tests.m2_runner import M2Run
    shape = gen.Mamba2Shape(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=8)
    r = M2Run(shape, 17, h0=gen.mamba2_random_state(shape, 17), sample=[0], conventional=False)
    r.decode(0)
    r.cache.ring_head[5] = 8                               # >= L
    before = r.cache.ckpt[5].clone()
    rx = r.cache.rec_x[5].clone()
    d = gen.mamba2_draft_inputs(shape, r.params, 17, 1, 4)
    rs.verify(r.cache, to_dev(d.dt), to_dev(d.x, torch.bfloat16), to_dev(d.B, torch.bfloat16),
              to_dev(d.C, torch.bfloat16))
    torch.cuda.synchronize()
    assert int(r.cache.err.item()) & rs.DEVERR_RING_META
    assert r.cache.ring_head[5].item() == 8 and r.cache.ring_len[5].item() == 1
    assert torch.equal(r.cache.ckpt[5], before) and torch.equal(r.cache.rec_x[5], rx)
    assert r.cache.ring_len[0].item() == 5 and not r.cache.arrive.any().item()
