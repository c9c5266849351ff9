"""The oracle pins must catch plausible mistakes.

Each case plants one slip in a copy of the oracle's update (on the CPU, by
monkeypatching) and checks that the pins above reject it.
"""
import numpy as np
import pytest

import oracle.gdn as gdn_mod
import oracle.mamba2 as m2_mod
from tests import test_oracle_gdn as gdn_pins
from tests import test_oracle_mamba2 as m2_pins


def _m2_mutants():
    def decay_after_input(self, h, dt, x, B, C):
        dt = np.asarray(dt, np.float64); x = np.asarray(x, np.float64)
        Bh = np.asarray(B, np.float64)[:, self.g]; Ch = np.asarray(C, np.float64)[:, self.g]
        a = np.exp(dt * self.A[None])
        h = a[:, :, None, None] * (h + (dt[:, :, None] * x)[..., None] * Bh[:, :, None, :])
        return h, np.einsum("bhpn,bhn->bhp", h, Ch) + self.D[None, :, None] * x

    def dropped_dt_on_input(self, h, dt, x, B, C):
        dt = np.asarray(dt, np.float64); x = np.asarray(x, np.float64)
        Bh = np.asarray(B, np.float64)[:, self.g]; Ch = np.asarray(C, np.float64)[:, self.g]
        a = np.exp(dt * self.A[None])
        h = a[:, :, None, None] * h + x[..., None] * Bh[:, :, None, :]
        return h, np.einsum("bhpn,bhn->bhp", h, Ch) + self.D[None, :, None] * x

    def swapped_B_C(self, h, dt, x, B, C):
        return m2_mod.Mamba2Stepwise._orig(self, h, dt, x, C, B)

    def wrong_group(self, h, dt, x, B, C):
        g = self.g
        self.g = np.arange(len(g)) % B.shape[1]
        try:
            return m2_mod.Mamba2Stepwise._orig(self, h, dt, x, B, C)
        finally:
            self.g = g

    def no_skip_term(self, h, dt, x, B, C):
        h, y = m2_mod.Mamba2Stepwise._orig(self, h, dt, x, B, C)
        return h, y - self.D[None, :, None] * np.asarray(x, np.float64)

    def output_before_update(self, h, dt, x, B, C):
        Ch = np.asarray(C, np.float64)[:, self.g]
        y = np.einsum("bhpn,bhn->bhp", h, Ch) + self.D[None, :, None] * np.asarray(x, np.float64)
        h, _ = m2_mod.Mamba2Stepwise._orig(self, h, dt, x, B, C)
        return h, y

    return [decay_after_input, dropped_dt_on_input, swapped_B_C, wrong_group,
            no_skip_term, output_before_update]


def _run_pins(module):
    failed = 0
    for name in dir(module):
        if name.startswith("test_"):
            try:
                getattr(module, name)()
            except AssertionError:
                failed += 1
    return failed


@pytest.mark.parametrize("mutant", _m2_mutants(), ids=lambda f: f.__name__)
def test_mamba2_pins_catch(monkeypatch, mutant):
    m2_mod.Mamba2Stepwise._orig = m2_mod.Mamba2Stepwise._update
    monkeypatch.setattr(m2_mod.Mamba2Stepwise, "_update", mutant)
    assert _run_pins(m2_pins) > 0


def _gdn_mutants():
    def sign_flip(self, S, q, k, v, alpha, beta):
        return gdn_mod.GDNStepwise._orig(self, S, q, k, -np.asarray(v), alpha, beta)

    def decay_outside(self, S, q, k, v, alpha, beta):
        q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
        a = np.asarray(alpha, np.float64)[:, :, None, None]; bt = np.asarray(beta, np.float64)[:, :, None, None]
        Sk = np.einsum("bhvk,bhk->bhv", S, k)
        S = a * (S - bt * Sk[..., None] * k[:, :, None, :] + bt * v[..., None] * k[:, :, None, :])
        return S, np.einsum("bhvk,bhk->bhv", S, q)

    def transposed_outer(self, S, q, k, v, alpha, beta):
        q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
        a = np.asarray(alpha, np.float64)[:, :, None, None]; bt = np.asarray(beta, np.float64)[:, :, None, None]
        kS = np.einsum("bhvk,bhv->bhk", S, k[..., :S.shape[2]]) if S.shape[2] == S.shape[3] else None
        if kS is None:
            raise AssertionError("shape")
        S = a * (S - bt * k[..., None] * kS[:, :, None, :]) + bt * v[..., None] * k[:, :, None, :]
        return S, np.einsum("bhvk,bhk->bhv", S, q)

    return [sign_flip, decay_outside, transposed_outer]


@pytest.mark.parametrize("mutant", _gdn_mutants(), ids=lambda f: f.__name__)
def test_gdn_pins_catch(monkeypatch, mutant):
    gdn_mod.GDNStepwise._orig = gdn_mod.GDNStepwise._update
    monkeypatch.setattr(gdn_mod.GDNStepwise, "_update", mutant)
    assert _run_pins(gdn_pins) > 0


def _gdn_verify_mutants():
    def drafts_not_causal(self, q, k, v, alpha, beta):
        T = np.asarray(alpha).shape[1]
        outs, states = [], []
        for i in range(T):                       # every draft scored from the checkpoint alone
            S, o = self._update(self.S, q[:, i], k[:, i], v[:, i], alpha[:, i], beta[:, i])
            outs.append(o)
            states.append(S)
        return np.stack(outs, axis=1), states

    def accept_off_by_one(self, states, accepted):
        new = self.S.copy()
        for b, a in enumerate(np.asarray(accepted)):
            if a > 0:
                new[b] = states[min(a, len(states) - 1)][b]
        self.S = new

    return [("verify", drafts_not_causal), ("accept", accept_off_by_one)]


@pytest.mark.parametrize("mutant", _gdn_verify_mutants(), ids=lambda m: m[1].__name__)
def test_gdn_verify_pins_catch(monkeypatch, mutant):
    attr, fn = mutant
    monkeypatch.setattr(gdn_mod.GDNStepwise, attr, fn)
    assert _run_pins(gdn_pins) > 0


def _nvfp4_mutants():
    import oracle.nvfp4 as nv

    def swapped_nibbles(codes):
        c = np.asarray(codes, np.uint8)
        return (c[..., 1::2] | (c[..., 0::2] << 4)).astype(np.uint8)

    def ties_away_from_zero(v):
        v = np.asarray(v, np.float32)
        a = np.abs(v.astype(np.float64))
        _, ex = np.frexp(a)
        q = np.ldexp(0.5, np.maximum(ex - 1, 0))
        val = np.minimum(np.floor(a / q + 0.5) * q, 6.0)
        mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
        code = np.abs(val[..., None] - mags).argmin(axis=-1)
        return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)

    def dropped_sign(v):
        return nv._orig_encode(np.abs(np.asarray(v, np.float32)))

    def row_target_448(h):
        old = nv.ROW_TARGET
        nv.ROW_TARGET = 448.0
        try:
            return nv._orig_quantize(h)
        finally:
            nv.ROW_TARGET = old

    def block_of_8(h):
        old = nv.BLOCK
        nv.BLOCK = 8
        try:
            return nv._orig_quantize(h)
        finally:
            nv.BLOCK = old

    def block_scale_from_row_max(h):
        h = np.asarray(h, np.float32)
        codes, sb, s_r = nv._orig_quantize(h)
        top = sb.max(axis=-1, keepdims=True)
        return codes, np.broadcast_to(top, sb.shape).copy(), s_r

    return [("pack_codes", swapped_nibbles), ("e2m1_encode", ties_away_from_zero),
            ("e2m1_encode", dropped_sign), ("quantize_rows", row_target_448),
            ("quantize_rows", block_of_8), ("quantize_rows", block_scale_from_row_max)]


@pytest.mark.parametrize("target,mutant", _nvfp4_mutants(), ids=lambda m: getattr(m, "__name__", str(m)))
def test_nvfp4_pins_catch(monkeypatch, target, mutant):
    import oracle.nvfp4 as nv
    from tests import test_oracle_nvfp4 as nv_pins
    nv._orig_encode = nv.e2m1_encode
    nv._orig_quantize = nv.quantize_rows
    monkeypatch.setattr(nv, target, mutant)
    failed = 0
    for name in dir(nv_pins):
        if name.startswith("test_"):
            try:
                getattr(nv_pins, name)()
            except (AssertionError, ValueError):      # a wrong value, or a wrong block count
                failed += 1
    assert failed > 0


def _f16sr_mutants():
    import oracle.f16sr as sr

    def philox_nine_rounds(ctr, key):
        c = np.asarray(ctr, np.uint64) & 0xFFFFFFFF
        k = np.asarray(key, np.uint64) & 0xFFFFFFFF
        c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
        k0, k1 = k[..., 0], k[..., 1]
        for rnd in range(9):
            if rnd > 0:
                k0 = (k0 + sr._W0) & 0xFFFFFFFF
                k1 = (k1 + sr._W1) & 0xFFFFFFFF
            p0, p1 = c0 * np.uint64(sr._M0), c2 * np.uint64(sr._M1)
            c0, c1, c2, c3 = (p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & np.uint64(0xFFFFFFFF), \
                (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & np.uint64(0xFFFFFFFF)
        return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)

    def halves_swapped(seed, slot, head, P, N):
        r = sr._orig_random16(seed, slot, head, P, N)
        return ((r >> 8) | (r << 8)) & 0xFFFF

    def round_to_nearest(v, r):
        with np.errstate(over="ignore"):                   # values above 65504 become inf here
            return np.asarray(v, np.float32).astype(np.float16)

    def round_up_on_equal(v, r):
        v = np.asarray(v, np.float32)
        return sr._orig_sr(v, np.asarray(r) - 1)           # r <= p * 65536

    def truncate(v, r):
        return sr._orig_sr(v, np.full(np.shape(v), 65535))

    return [("philox4x32_10", philox_nine_rounds), ("random16", halves_swapped),
            ("sr_f16", round_to_nearest), ("sr_f16", round_up_on_equal), ("sr_f16", truncate)]


@pytest.mark.parametrize("target,mutant", _f16sr_mutants(), ids=lambda m: getattr(m, "__name__", str(m)))
def test_f16sr_pins_catch(monkeypatch, target, mutant):
    import oracle.f16sr as sr
    from tests import test_oracle_f16sr as pins
    sr._orig_random16 = sr.random16
    sr._orig_sr = sr.sr_f16
    monkeypatch.setattr(sr, target, mutant)
    assert _run_pins(pins) > 0
