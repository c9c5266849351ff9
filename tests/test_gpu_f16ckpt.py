"""FP16 checkpoint with stochastic rounding at every flush, against the oracle
(oracle.f16sr).

* Exact folds: with a decay of exactly 1 (A so small that exp(A S) rounds to
  1 in float32), dt a power of two, x and B of few bits and an FP16
  checkpoint, every fold is exact in float32, so the kernel and the oracle
  round the same float32 value with the same random integers: the FP16
  checkpoint after the flush is bit for bit the oracle's, for the fused flush
  (persistent and per-tile kernels), the standalone flush and the verify
  pre-flush.
* Real inputs: between flushes y is the oracle's stepwise y from the FP16
  checkpoint (float32 gate); at a flush every element is the oracle's rounding
  of the exact fold or its FP16 neighbour (the float32 values the two round
  differ in the last bits, which moves a decision only rarely), and the
  rounding errors average out (unbiased).
"""
import numpy as np
import pytest
import torch

from oracle.f16sr import Mamba2F16SR, random16, sr_f16
from oracle.mamba2 import Mamba2Stepwise
from oracle.nvfp4 import head_copy
from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL, assert_close, to_dev

pytestmark = pytest.mark.gpu

TINY_A = -(2.0 ** -40)          # exp(TINY_A * S) rounds to 1.0 in float32 for S < 2^10


def _f16_state(shape, seed, floor=2.0 ** -6):
    """FP16 checkpoint values of magnitude about 4 (FP16 steps 2^-9..2^-8, finer
    than most fold terms), none below `floor`, so that a fold spans at most ~21
    bits and stays exact in float32."""
    h = gen.mamba2_random_state(shape, seed, std=4.0).astype(np.float16)
    return np.where(np.abs(h.astype(np.float32)) < floor, np.float16(0), h)


def _exact_step(shape, rng, T=None):
    lead = (shape.batch,) if T is None else (shape.batch, T)
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    dt = np.full(lead + (H,), 2.0 ** -7, np.float32)
    x = rng.choice([-2.0, -1.0, -0.5, -0.25, 0.25, 0.5, 1.0, 2.0], size=lead + (H, P)).astype(np.float32)
    B = rng.choice([-1.0, -0.75, -0.5, -0.25, 0.25, 0.5, 0.75, 1.0], size=lead + (G, N)).astype(np.float32)
    C = gen.round_bf16((rng.standard_normal(lead + (G, N)) / np.sqrt(N)).astype(np.float32))
    return gen.Mamba2Step(dt=dt, x=x, B=B, C=C)


def _cache(shape, h0_f16, A, D, read_copy=0, seed0=1000):
    from ssm_decode_state_gb300 import replayssm as rs
    dims = rs.mamba2_dims(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L,
                          read_copy=read_copy, ckpt_f16=True)
    c = rs.mamba2_cache(dims, torch.from_numpy(np.asarray(A, np.float32)), torch.from_numpy(np.asarray(D, np.float32)),
                        ckpt=torch.from_numpy(h0_f16).cuda())
    c.sr_seed = seed0
    return rs, c


def _dev(st):
    return (to_dev(st.dt), to_dev(st.x, torch.bfloat16), to_dev(st.B, torch.bfloat16), to_dev(st.C, torch.bfloat16))


def _exact_fold(h_f16, steps, g):
    """h + sum_j dt_j x_j B_j^T in float64 (exact here), [b, H, P, N]."""
    v = h_f16.astype(np.float64)
    for st in steps:
        v = v + (st.dt[:, :, None] * st.x)[..., None] * st.B[:, g][:, :, None, :]
    return v


def _sr_expected(v, seed, seqs, slots=None):
    b_, H, P, N = v.shape
    out = np.empty(v.shape, np.float16)
    for b in seqs:
        s = b if slots is None else int(slots[b])
        for h in range(H):
            out[b, h] = sr_f16(v[b, h].astype(np.float32), random16(seed, s, h, P, N))
    return out


@pytest.mark.parametrize("shape", [
    gen.Mamba2Shape(batch=2, nheads=128, headdim=64, dstate=128, ngroups=8, L=4),     # persistent, 2 heads per item
    gen.Mamba2Shape(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=4),   # persistent, 8 heads per item
    gen.Mamba2Shape(batch=3, nheads=6, headdim=32, dstate=64, ngroups=3, L=5),        # per-tile
], ids=["persistent_b2", "persistent_b128", "per_tile"])
def test_fused_flush_rounds_like_the_oracle_bitwise(shape):
    rng = np.random.default_rng(11)
    h0 = _f16_state(shape, 11)
    A = np.full(shape.nheads, TINY_A)
    D = rng.standard_normal(shape.nheads)
    rs, c = _cache(shape, h0, A, D)
    g = np.arange(shape.nheads) // (shape.nheads // shape.ngroups)
    orc = Mamba2Stepwise(A, D, shape.ngroups, h0.astype(np.float64))
    steps, seed = [], None
    for t in range(shape.L):
        st = _exact_step(shape, rng)
        seed = c.sr_seed
        y = rs.decode(c, *_dev(st))
        yo = orc.step(st.dt, st.x, st.B, st.C)
        assert_close(y.cpu().numpy(), yo, f"y at step {t}", RTOL)
        steps.append(st)
    assert not c.ring_len.any().item()                   # the L-th token folded
    seqs = range(shape.batch) if shape.batch <= 8 else [0, 77, shape.batch - 1]
    want = _sr_expected(_exact_fold(h0, steps, g), seed, seqs)
    got = c.ckpt.cpu().numpy()
    for b in seqs:
        np.testing.assert_array_equal(got[b].view(np.uint16), want[b].view(np.uint16))
    # the rounding did something: many elements are not FP16 values of the exact fold
    v = _exact_fold(h0, steps, g)[list(seqs)]
    assert np.mean(v.astype(np.float16).astype(np.float64) != v) > 0.3
    assert int(c.err.item()) == 0


def test_standalone_flush_and_verify_preflush_bitwise():
    """Masked standalone flush after 2 tokens, then a verify whose drafts do
    not fit the ring (pre-flush of the buffered records), both exact."""
    shape = gen.Mamba2Shape(batch=4, nheads=8, headdim=32, dstate=64, ngroups=2, L=6)
    rng = np.random.default_rng(12)
    h0 = _f16_state(shape, 12)
    A, D = np.full(shape.nheads, TINY_A), rng.standard_normal(shape.nheads)
    rs, c = _cache(shape, h0, A, D)
    g = np.arange(shape.nheads) // (shape.nheads // shape.ngroups)
    steps = [_exact_step(shape, rng) for _ in range(2)]
    for st in steps:
        rs.decode(c, *_dev(st))
    mask = np.array([1, 0, 1, 0], np.uint8)
    seed = c.sr_seed
    rs.flush(c, torch.from_numpy(mask).cuda())
    v = _exact_fold(h0, steps, g)
    want = _sr_expected(v, seed, [0, 2])
    got = c.ckpt.cpu().numpy()
    for b in (0, 2):
        np.testing.assert_array_equal(got[b].view(np.uint16), want[b].view(np.uint16))
    for b in (1, 3):
        np.testing.assert_array_equal(got[b], h0[b])
    # rows 1, 3 hold 2 records; 3 more tokens, then 3 drafts: 5 + 3 > 6 pre-flushes them
    more = [_exact_step(shape, rng) for _ in range(3)]
    for st in more:
        rs.decode(c, *_dev(st))
    ck_before = c.ckpt.cpu().numpy()
    T = 3
    d = _exact_step(shape, rng, T)
    seed = c.sr_seed
    rs.verify(c, *_dev(d))
    got = c.ckpt.cpu().numpy()
    v13 = _exact_fold(h0, steps + more, g)
    want13 = _sr_expected(v13, seed, [1, 3])
    for b in (1, 3):
        np.testing.assert_array_equal(got[b].view(np.uint16), want13[b].view(np.uint16))
    # rows 0, 2 held 3 records: 3 + 3 <= 6, no pre-flush
    for b in (0, 2):
        np.testing.assert_array_equal(got[b], ck_before[b])
    assert int(c.err.item()) == 0


def test_requant_from_fp16_checkpoint():
    """Both read copies built from an FP16 checkpoint equal the oracle's
    quantisation of its values, byte for byte."""
    from oracle.fp8 import quantize_rows
    shape = gen.Mamba2Shape(batch=3, nheads=4, headdim=64, dstate=128, ngroups=1, L=16)
    h0 = _f16_state(shape, 13, floor=0.0)
    for rc in (1, 2):
        rs, c = _cache(shape, h0, np.full(4, -1.0), np.zeros(4), read_copy=rc)
        rs.requant(c)
        if rc == 1:
            codes, scale = quantize_rows(h0.astype(np.float32))
            np.testing.assert_array_equal(c.ckpt_q.cpu().numpy(), codes)
        else:
            stored, scale = head_copy(h0.astype(np.float32))
            np.testing.assert_array_equal(c.ckpt_q.cpu().numpy(), stored)
        np.testing.assert_array_equal(c.ckpt_scale.cpu().numpy(), scale)


class _F16Run:
    """Real inputs: the kernel's FP16-checkpoint cache and the oracle on the
    sampled sequences, the oracle re-synchronised to the kernel's checkpoint at
    the start of every flush window."""

    def __init__(self, shape, seed, sample, read_copy=0):
        self.shape, self.seed, self.sample = shape, seed, list(sample)
        self.prm = gen.mamba2_params(shape, seed)
        h0 = gen.mamba2_random_state(shape, seed).astype(np.float16)
        self.rs, self.c = _cache(shape, h0, self.prm.A, self.prm.D, read_copy=read_copy, seed0=seed * 7919)
        if read_copy:
            self.rs.requant(self.c)
        self.orc = Mamba2F16SR(self.prm.A, self.prm.D, shape.ngroups, h0[self.sample], shape.L, slots=self.sample)
        self.g = np.arange(shape.nheads) // (shape.nheads // shape.ngroups)
        self.z = []                    # (kernel - oracle rounding) / step, every flushed element
        self.mismatch = [0, 0]

    def step(self, t):
        s = self.sample
        st = gen.mamba2_step_inputs(self.shape, self.prm, self.seed, t)
        seed = self.c.sr_seed
        y = self.rs.decode(self.c, *_dev(st)).cpu().numpy()[s]
        exact_before = self.orc.h.copy()
        folding = self.orc.len[0] + 1 >= self.shape.L
        yo = self.orc.decode(st.dt[s], st.x[s], st.B[s], st.C[s], seed)
        assert_close(y, yo, f"y at step {t}", RTOL)
        if folding:
            got = self.c.ckpt[s].cpu().numpy().astype(np.float64)
            want = self.orc.h
            # the exact fold the oracle rounded
            sw = Mamba2Stepwise(self.prm.A, self.prm.D, self.shape.ngroups, exact_before)
            sw.step(st.dt[s], st.x[s], st.B[s], st.C[s])
            v = sw.h
            step_ = np.maximum(np.abs(v.astype(np.float16).astype(np.float64)) * 2.0 ** -10, 2.0 ** -24)
            diff = np.abs(got - want)
            assert np.all((diff == 0) | (diff <= 2.0 * step_)), "kernel rounding is not a neighbour of the oracle's"
            self.mismatch[0] += int(np.sum(diff != 0))
            self.mismatch[1] += diff.size
            self.z.append(((got - v) / step_).ravel())
            self.orc.h = got.copy()                      # continue from the kernel's checkpoint
        return y

    def finish(self):
        assert self.mismatch[0] <= 0.01 * self.mismatch[1], self.mismatch
        z = np.concatenate(self.z)
        # SR error per element has mean 0 and variance p(1-p) <= 1/4 (in steps)
        assert abs(z.mean()) <= 5 * 0.5 / np.sqrt(z.size), z.mean()
        assert int(self.c.err.item()) == 0


def test_fp16_checkpoint_decode_b256():
    """Serving shape at batch 256, 3 flush windows; the oracle follows 2 sequences."""
    shape = gen.Mamba2Shape(batch=256, nheads=128, headdim=64, dstate=128, ngroups=8, L=16)
    r = _F16Run(shape, 21, [5, 250])
    for t in range(3 * shape.L):
        r.step(t)
    r.finish()


def test_fp16_checkpoint_decode_per_tile():
    shape = gen.Mamba2Shape(batch=5, nheads=6, headdim=32, dstate=64, ngroups=3, L=8)
    r = _F16Run(shape, 22, [0, 1, 2, 3, 4])
    for t in range(4 * shape.L):
        r.step(t)
    r.finish()


def test_fp16_checkpoint_with_nvfp4_reads():
    """NVFP4 reads of an FP16 recurrence (the pairing the pages report): after
    every flush the copy is the oracle's quantisation of the new FP16
    checkpoint, byte for byte."""
    shape = gen.Mamba2Shape(batch=16, nheads=128, headdim=64, dstate=128, ngroups=8, L=8)
    prm = gen.mamba2_params(shape, 23)
    h0 = gen.mamba2_random_state(shape, 23).astype(np.float16)
    rs, c = _cache(shape, h0, prm.A, prm.D, read_copy=2)
    rs.requant(c)
    for t in range(2 * shape.L):
        st = gen.mamba2_step_inputs(shape, prm, 23, t)
        rs.decode(c, *_dev(st))
        if (t + 1) % shape.L == 0:
            stored, s_r = head_copy(c.ckpt.cpu().numpy().astype(np.float32))
            np.testing.assert_array_equal(c.ckpt_q.cpu().numpy(), stored)
            np.testing.assert_array_equal(c.ckpt_scale.cpu().numpy(), s_r)
    assert int(c.err.item()) == 0
