"""NVFP4 read copy (E2M1 codes, an E4M3 scale per 16 columns, a float32 scale
per row) against the oracle (oracle.nvfp4).

* The copy the kernels write (requant, fused flush, standalone flush, verify
  pre-flush) equals the oracle's quantisation of the kernel's own FP32
  checkpoint, byte for byte: the codes are integer decisions taken in float32
  on both sides.
* Reads: on non-flush steps y equals the oracle's FP32 output plus
  exp(A S) (x_hat - h_c) . C_t, x_hat the oracle's decoding of the copy the
  kernel read, within the float32 gate; arbitrary code bytes (all 16 E2M1
  codes, block scales over the E4M3 range) decode exactly.
"""
import numpy as np
import pytest
import torch

from oracle.mamba2 import Mamba2Stepwise
from oracle.nvfp4 import head_copy, head_dequantize
from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL, assert_close, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _cache(shape, seed, h0, capacity=0):
    from ssm_decode_state_gb300 import replayssm as rs
    prm = gen.mamba2_params(shape, seed)
    dims = rs.mamba2_dims(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L,
                          read_copy=2)
    c = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D), ckpt=to_dev(h0))
    return rs, prm, c


def _check_copy(c, seqs=None):
    """The stored copy of the given sequences equals the oracle's quantisation
    of the kernel's FP32 checkpoint, byte for byte."""
    idx = slice(None) if seqs is None else list(seqs)
    ck = c.ckpt[idx].cpu().numpy()
    stored, s_r = head_copy(ck)
    np.testing.assert_array_equal(c.ckpt_q[idx].cpu().numpy(), stored)
    np.testing.assert_array_equal(c.ckpt_scale[idx].cpu().numpy(), s_r)


@pytest.mark.parametrize("P,N", [(64, 128), (32, 64), (16, 16)])
def test_requant_matches_oracle_bytewise(P, N):
    """Codes, block scales and row scales of the whole cache, including a zero
    row, a row of negative zeros, a row too small for the scales, a block with
    a subnormal E4M3 scale, and saturating values."""
    shape = gen.Mamba2Shape(batch=3, nheads=4, headdim=P, dstate=N, ngroups=1, L=16)
    h0 = gen.mamba2_random_state(shape, 92)
    h0[0, 0, 3] = 0.0
    h0[0, 1, 2] = -0.0
    h0[1, 2, 5] *= 1e-41
    h0[1, 3, 1, :16] *= 1e-5                 # block scale below the smallest normal E4M3
    h0[2, 1, 7, :5] = 1e6
    h0[2, 2, 0, 8:] = -3e-3
    rs, _, c = _cache(shape, 92, h0)
    rs.requant(c)
    _check_copy(c)


def _exact_decode(shape, seed):
    """Random code bytes (every nibble value), block scales drawn over the
    finite E4M3 codes (subnormal ones included), random row scales: one
    non-flush decode step reads the copy; y against the oracle stepping from
    the decoded values."""
    rs, prm, c = _cache(shape, seed, np.zeros((shape.batch, shape.nheads, shape.headdim, shape.dstate),
                                             np.float32))
    P, N = shape.headdim, shape.dstate
    rng = np.random.default_rng(seed)
    nb = P * N // 2
    stored = rng.integers(0, 256, size=(shape.batch, shape.nheads, nb + P * N // 16), dtype=np.uint8)
    sbc = rng.integers(0, 0x7F, size=(shape.batch, shape.nheads, P * N // 16), dtype=np.uint8)   # finite, >= 0
    stored[..., nb:] = sbc
    s_r = (rng.uniform(0.5, 2.0, size=(shape.batch, shape.nheads, P)) * 2.0 ** -8).astype(np.float32)
    c.ckpt_q.copy_(torch.from_numpy(stored))
    c.ckpt_scale.copy_(torch.from_numpy(s_r))
    sm = sorted({0, shape.batch // 2, shape.batch - 1})
    xhat = head_dequantize(stored[sm], s_r[sm], P, N)         # float64, exact
    orc = Mamba2Stepwise(prm.A, prm.D, shape.ngroups, xhat)
    st = gen.mamba2_step_inputs(shape, prm, seed, 0)
    y = rs.decode(c, to_dev(st.dt), to_dev(st.x, torch.bfloat16), to_dev(st.B, torch.bfloat16),
                  to_dev(st.C, torch.bfloat16))
    yo = orc.step(st.dt[sm], st.x[sm], st.B[sm], st.C[sm])
    # float32 accumulation bound of the checkpoint term: each lane sums 16
    # products of exact values, then 3 levels of a tree over the block lanes,
    # the block scale and the row scale: at most 32 roundings of 2^-24 relative
    # to sum |x_hat C|; random codes make that sum far larger than y
    g = np.arange(shape.nheads) // (shape.nheads // shape.ngroups)
    mag = np.einsum("shpn,shn->shp", np.abs(xhat), np.abs(st.C[sm][:, g].astype(np.float64)))
    decay = np.exp(prm.A[None].astype(np.float64) * st.dt[sm].astype(np.float64))
    tau = 1e-2 * np.sqrt(np.mean(yo ** 2))
    bound = 32 * 2.0 ** -24 * decay[..., None] * mag + 1e-5 * np.maximum(np.abs(yo), tau)
    err = np.abs(y.cpu().numpy()[sm] - yo)
    assert np.all(err <= bound), f"y from arbitrary NVFP4 codes: worst err / bound {np.max(err / bound):.3f}"
    assert_close(y.cpu().numpy()[sm], yo, "y from arbitrary NVFP4 codes", RTOL)
    assert int(c.err.item()) == 0


def test_exact_decode_persistent():
    """Batch 120 at 128 heads: 8 heads per work item, 4 per NVFP4 stage."""
    _exact_decode(gen.Mamba2Shape(batch=120, nheads=128, headdim=64, dstate=128, ngroups=8, L=16), 31)


def test_exact_decode_per_tile():
    _exact_decode(gen.Mamba2Shape(batch=3, nheads=8, headdim=32, dstate=64, ngroups=2, L=8), 32)


@pytest.mark.parametrize("batch", [1, 2, 5])
def test_exact_decode_small_batches(batch):
    """Smaller batches run the persistent kernel with 1 (batch 1), 2 (batch 2)
    or 4 (batch 5) heads per work item."""
    _exact_decode(gen.Mamba2Shape(batch=batch, nheads=128, headdim=64, dstate=128, ngroups=8, L=16), 40 + batch)


class _NV4Run:
    """An NVFP4-read cache and an FP32-read cache on the same inputs; the oracle
    follows the sampled sequences."""

    def __init__(self, shape, seed, sample):
        from tests.m2_runner import M2Run
        self.shape, self.seed, self.sample = shape, seed, list(sample)
        h0 = gen.mamba2_random_state(shape, seed)
        self.r4 = M2Run(shape, seed, h0=h0, read_copy=2, sample=sample, conventional=False)
        self.r32 = M2Run(shape, seed, h0=h0, read_copy=0, sample=[0], conventional=False, h0_sample=h0[:1])
        self.g = np.arange(shape.nheads) // (shape.nheads // shape.ngroups)
        self.dts = []                                  # dt of the records since the last flush

    def step(self, t):
        from ssm_decode_state_gb300 import replayssm as rs
        r4, s = self.r4, self.sample
        st = gen.mamba2_step_inputs(self.shape, r4.params, self.seed, t)
        dt, x, B, C = r4.dev_inputs(st)
        ln = int(r4.cache.ring_len[s[0]].item())
        ck = r4.cache.ckpt[s].cpu().numpy()
        stored = r4.cache.ckpt_q[s].cpu().numpy()
        s_r = r4.cache.ckpt_scale[s].cpu().numpy()
        y4 = rs.decode(r4.cache, dt, x, B, C).cpu().numpy()[s]
        rs.decode(self.r32.cache, dt, x, B, C)
        yo = r4.oracle.step(*r4._slice(st))
        r4.ring.decode([t] * self.shape.batch)
        self.dts.append(st.dt[s].astype(np.float64))
        if ln + 1 < self.shape.L:
            S = np.sum(self.dts, axis=0)
            decay = np.exp(r4.params.A[None].astype(np.float64) * S)
            xhat = head_dequantize(stored, s_r, self.shape.headdim, self.shape.dstate)
            dC = np.einsum("shpn,shn->shp", xhat - ck.astype(np.float64), st.C[s][:, self.g].astype(np.float64))
            want = yo + decay[..., None] * dC
            e = assert_close(y4, want, f"NVFP4 read y at step {t}", RTOL)
            # the copy is really read: its rounding moves y far beyond the gate
            assert rel_err(y4, yo) > 100 * RTOL
            return e
        # flush step: y from the FP32 values; the FP32 checkpoint equals the
        # FP32-read run's; the re-quantised copy is the oracle's quantisation
        self.dts = []
        assert_close(y4, yo, f"flush-step y at step {t}", RTOL)
        np.testing.assert_array_equal(r4.cache.ckpt[s].cpu().numpy(), self.r32.cache.ckpt[s].cpu().numpy())
        _check_copy(r4.cache, s)
        return 0.0


def test_nvfp4_read_decode_b256():
    """Serving shape at batch 256 (H 128, P 64, N 128, G 8, L 16), 4 flush
    windows; the oracle follows sequences 7 and 200."""
    shape = gen.Mamba2Shape(batch=256, nheads=128, headdim=64, dstate=128, ngroups=8, L=16)
    r = _NV4Run(shape, 77, [7, 200])
    for t in range(4 * shape.L):
        r.step(t)
    assert int(r.r4.cache.err.item()) == 0


def test_nvfp4_read_decode_per_tile():
    """Non-serving shape (per-tile kernel), ragged batch, 3 flush windows."""
    shape = gen.Mamba2Shape(batch=5, nheads=6, headdim=32, dstate=64, ngroups=3, L=8)
    r = _NV4Run(shape, 78, [0, 4])
    for t in range(3 * shape.L):
        r.step(t)


@pytest.mark.parametrize("batch,T", [(4, 3), (128, 4)], ids=["per_tile", "persistent"])
def test_nvfp4_verify_preflush_and_flush(batch, T):
    """A verify that pre-flushes re-quantises the copy of the folded sequences,
    and so does the masked standalone flush: byte-exact against the oracle's
    quantisation of the new checkpoint."""
    from ssm_decode_state_gb300 import replayssm as rs
    P, N = (64, 128) if batch >= 128 else (32, 64)
    shape = gen.Mamba2Shape(batch=batch, nheads=128 if batch >= 128 else 8, headdim=P, dstate=N,
                            ngroups=8 if batch >= 128 else 2, L=8)
    h0 = gen.mamba2_random_state(shape, 79)
    _, prm, c = _cache(shape, 79, h0)
    rs.requant(c)
    seqs = [0, batch // 2, batch - 1]
    for t in range(6):
        d = gen.mamba2_draft_inputs(shape, prm, 79, t, T)
        rs.verify(c, to_dev(d.dt), to_dev(d.x, torch.bfloat16), to_dev(d.B, torch.bfloat16),
                  to_dev(d.C, torch.bfloat16))
        rs.rollback(c, T, torch.from_numpy(gen.accepted_counts(batch, T, 79, t)).cuda())
        _check_copy(c, seqs)
    mask = torch.from_numpy((np.arange(batch) % 2 == 0).astype(np.uint8)).cuda()
    rs.flush(c, mask)
    _check_copy(c, seqs)
    assert int(c.err.item()) == 0
