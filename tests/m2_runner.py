"""Drives the CUDA Mamba-2 paths and the oracle side by side on one workload.

The GPU runs every sequence of the batch; the oracle follows the sequences in
``sample`` (all of them for small cases).  Every step compares y, the ring
pointers of every sequence (bit-exact against the integer ring model), and at
flush steps the checkpoint of the sampled sequences.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle.mamba2 import Mamba2Stepwise
from oracle.ring import RingModel
from ssm_decode_state_gb300 import inputs as gen
from ssm_decode_state_gb300 import replayssm as rs
from tests.helpers import RTOL_INPLACE, assert_close, io_dtype, rel_err, to_dev


class M2Run:
    def __init__(self, shape: gen.Mamba2Shape, seed: int, h0: np.ndarray | None = None,
                 read_copy: int = 0, sample=None, conventional: bool = True,
                 h0_sample: np.ndarray | None = None):
        self.shape, self.seed = shape, seed
        self.params = gen.mamba2_params(shape, seed)
        b = shape.batch
        self.sample = np.arange(b) if sample is None else np.asarray(sample)
        self.dims = rs.mamba2_dims(b, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                                   shape.L, read_copy, shape.bf16_io)
        A = torch.from_numpy(self.params.A)
        D = torch.from_numpy(self.params.D)
        if h0 is None:
            h0 = np.zeros((b, shape.nheads, shape.headdim, shape.dstate), np.float32)
        ck = to_dev(h0)
        self.cache = rs.mamba2_cache(self.dims, A, D, ckpt=ck)
        self.conv = ck.clone() if conventional else None
        if h0_sample is None:
            h0_sample = h0[self.sample]
        self.oracle = Mamba2Stepwise(self.params.A, self.params.D, shape.ngroups, h0_sample)
        self.ring = RingModel(b, shape.L)
        self.tokens = {}          # tag -> step inputs (numpy), for record checks
        self.max_err = {"replay": 0.0, "conventional": 0.0, "ckpt": 0.0}
        if read_copy:
            rs.requant(self.cache)

    def _keep(self, step, st):
        self.tokens[step] = st
        live = {t if not isinstance(t, tuple) else t[0]
                for s in self.ring.seqs for t in s.tags}
        for k in list(self.tokens):
            if k not in live and k != step:
                del self.tokens[k]

    # ------------------------------------------------------------------ inputs
    def dev_inputs(self, st: gen.Mamba2Step):
        io = io_dtype(self.shape.bf16_io)
        return (to_dev(st.dt), to_dev(st.x, io), to_dev(st.B, io), to_dev(st.C, io))

    def _slice(self, st: gen.Mamba2Step):
        s = self.sample
        return st.dt[s], st.x[s], st.B[s], st.C[s]

    # --------------------------------------------------------------- operations
    def prefill_conventional(self, steps):
        """Stepwise prefill through the conventional kernel; the result becomes
        the replay checkpoint (ring empty)."""
        for t in steps:
            st = gen.mamba2_step_inputs(self.shape, self.params, self.seed, t)
            dt, x, B, C = self.dev_inputs(st)
            rs.conventional_decode(self.dims, self.conv, self.cache.A, self.cache.D, dt, x, B, C)
            self.oracle.step(*self._slice(st))
        self.cache.ckpt.copy_(self.conv)
        if self.dims.read_copy:
            rs.requant(self.cache)

    def decode(self, step: int, check=True, rtol=1e-4):
        st = gen.mamba2_step_inputs(self.shape, self.params, self.seed, step)
        dt, x, B, C = self.dev_inputs(st)
        y = rs.decode(self.cache, dt, x, B, C)
        yc = rs.conventional_decode(self.dims, self.conv, self.cache.A, self.cache.D, dt, x, B, C) \
            if self.conv is not None else None
        yo = self.oracle.step(*self._slice(st))
        folded = self.ring.decode([step] * self.shape.batch)
        self._keep(step, st)
        if check:
            s = self.sample
            e = assert_close(y.cpu().numpy()[s], yo, f"replay y step {step}", rtol)
            self.max_err["replay"] = max(self.max_err["replay"], e)
            if yc is not None:
                e = assert_close(yc.cpu().numpy()[s], yo, f"conventional y step {step}", RTOL_INPLACE)
                self.max_err["conventional"] = max(self.max_err["conventional"], e)
            self.check_ring()
            if any(f is not None for f in folded):
                self.check_ckpt(step, [i for i, f in enumerate(folded) if f is not None])
        return y, yo, folded

    def check_ring(self):
        np.testing.assert_array_equal(self.cache.ring_head.cpu().numpy(), self.ring.heads())
        np.testing.assert_array_equal(self.cache.ring_len.cpu().numpy(), self.ring.lens())
        assert int(self.cache.err.item()) == 0
        assert not self.cache.arrive.any().item()

    def check_ckpt(self, step, seqs=None, rtol=1e-4):
        ck = self.cache.ckpt.cpu().numpy()
        for i, b in enumerate(self.sample):
            if seqs is not None and b not in seqs:
                continue
            e = rel_err(ck[b], self.oracle.h[i])
            assert e <= rtol, f"checkpoint of seq {b} after step {step}: {e:.3e}"
            self.max_err["ckpt"] = max(self.max_err["ckpt"], e)

    def check_records(self, seqs=None):
        """Buffered records in the ring equal the inputs of the buffered tokens,
        bit for bit."""
        shp = self.shape
        rdt = self.cache.rec_dt.cpu().numpy()
        rx = self.cache.rec_x.float().cpu().numpy()
        rB = self.cache.rec_B.float().cpu().numpy()
        rC = self.cache.rec_C.float().cpu().numpy() if self.cache.rec_C is not None else None
        for b in (range(shp.batch) if seqs is None else seqs):
            for slot, tag in self.ring.seqs[b].slots().items():
                st = tag_inputs(self.tokens, tag)
                np.testing.assert_array_equal(rdt[b, :, slot], st.dt[b])
                np.testing.assert_array_equal(rx[b, :, slot], st.x[b])
                np.testing.assert_array_equal(rB[b, :, slot], st.B[b])
                if rC is not None:
                    np.testing.assert_array_equal(rC[b, :, slot], st.C[b])


def tag_inputs(tokens, tag):
    """A tag is a decode step id, or (step, i) for draft i of a verify step."""
    if isinstance(tag, tuple):
        st = tokens[tag[0]]
        i = tag[1]
        return gen.Mamba2Step(dt=st.dt[:, i], x=st.x[:, i], B=st.B[:, i], C=st.C[:, i])
    return tokens[tag]
