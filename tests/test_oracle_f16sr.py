"""Pins of the FP16 stochastic-rounding recurrence oracle (oracle.f16sr)."""
import json
import os

import numpy as np

import oracle.f16sr as sr
from oracle.mamba2 import Mamba2Stepwise
from ssm_decode_state_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def _all_f16_positive() -> np.ndarray:
    """Every finite non-negative FP16 value, ascending (from the bit patterns)."""
    return np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)


def test_philox_known_answers():
    with open(GOLDEN) as f:
        kat = json.load(f)
    for v in kat["vectors"]:
        ctr = np.array([int(w, 16) for w in v["ctr"]], np.uint64)
        key = np.array([int(w, 16) for w in v["key"]], np.uint64)
        got = sr.philox4x32_10(ctr, key)
        assert [f"{int(w):08x}" for w in got] == v["out"], v


def test_random16_element_mapping():
    """Element (p, n) of a head takes half n mod 2 of word (n mod 8) / 2 of the
    Philox output for counter (n / 8, p, head, slot), checked one call at a time."""
    seed, slot, head, P, N = 0x1234_5678_9ABC_DEF0, 7, 3, 4, 16
    r = sr.random16(seed, slot, head, P, N)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint64)
    for p in range(P):
        for n in range(N):
            out = sr.philox4x32_10(np.array([n // 8, p, head, slot], np.uint64), key)
            w = int(out[(n % 8) // 2])
            assert int(r[p, n]) == (w >> (16 * (n % 2))) & 0xFFFF


def test_exact_values_are_kept():
    """An FP16 value rounds to itself whatever the random integer."""
    v = _all_f16_positive()[::7]
    v = np.concatenate([v, -v]).astype(np.float32)
    for r in (0, 1, 12345, 65535):
        np.testing.assert_array_equal(sr.sr_f16(v, np.full(v.shape, r)).astype(np.float32), v)


def test_result_brackets_the_value():
    """The result is the FP16 neighbour below |v| or the one above (found by a
    search over all FP16 values), never anything else; above 65504 it saturates."""
    grid = _all_f16_positive()
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 5, 20000),
                        rng.uniform(6e4, 7e4, 200)]).astype(np.float32)
    a = np.abs(v.astype(np.float64))
    i = np.searchsorted(grid, np.minimum(a, 65504.0), side="right") - 1
    lo, hi = grid[i], grid[np.minimum(i + 1, len(grid) - 1)]
    res = np.abs(sr.sr_f16(v, rng.integers(0, 65536, v.shape)).astype(np.float64))
    ok = (res == lo) | (res == hi) | ((a >= 65504.0) & (res == 65504.0))
    assert ok.all()
    assert np.all(np.signbit(sr.sr_f16(v, np.zeros(v.shape))) == np.signbit(v))


def test_round_up_probability_is_exact():
    """Over all 65536 random integers, the share rounding up equals the fraction
    of the step (a - lo) / (hi - lo), exactly, for values in the normal FP16
    range; within 2^-16 below it."""
    grid = _all_f16_positive()
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.uniform(2.0 ** -14, 3e4, 24), rng.uniform(0, 2.0 ** -14, 8)]).astype(np.float32)
    r = np.arange(65536)
    for x in v:
        a = float(x)
        i = np.searchsorted(grid, a, side="right") - 1
        lo, hi = grid[i], grid[i + 1]
        up = np.mean(sr.sr_f16(np.full(65536, x), r).astype(np.float64) == hi)
        frac = (a - lo) / (hi - lo)
        if a >= 2.0 ** -14:
            assert up == frac, (a, up, frac)
        else:
            assert abs(up - frac) <= 2.0 ** -16, (a, up, frac)


def test_unbiased_over_seeds():
    """The mean over seeds of the rounded values is the float32 value (the
    error of a mean of K roundings shrinks as 1/sqrt(K))."""
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((8, 16)) * 0.1).astype(np.float32)
    acc = np.zeros(v.shape)
    K = 400
    for seed in range(K):
        acc += sr.sr_f16(v, sr.random16(seed, 0, 0, 8, 16)).astype(np.float64)
    step = np.abs(v.astype(np.float64)) * 2.0 ** -10
    assert np.all(np.abs(acc / K - v) <= 6 * step / np.sqrt(K) + 1e-12)


def test_recurrence_folds_at_the_ring_capacity():
    """Between flushes the state is the exact stepwise state from the FP16
    checkpoint; at the L-th token it becomes FP16 values within one step of the
    exact state, and averaged over seeds the folded state is the exact one."""
    shape = gen.Mamba2Shape(batch=2, nheads=2, headdim=8, dstate=16, ngroups=1, L=4)
    prm = gen.mamba2_params(shape, 6)
    h0 = gen.mamba2_random_state(shape, 6).astype(np.float16)
    mean = np.zeros(h0.shape)
    K = 64
    for seed in range(K):
        o = sr.Mamba2F16SR(prm.A, prm.D, 1, h0, shape.L)
        r = Mamba2Stepwise(prm.A, prm.D, 1, h0.astype(np.float64))
        for t in range(shape.L):
            st = gen.mamba2_step_inputs(shape, prm, 6, t)
            y = o.decode(st.dt, st.x, st.B, st.C, seed)
            yr = r.step(st.dt, st.x, st.B, st.C)
            np.testing.assert_allclose(y, yr, rtol=1e-12, atol=1e-15)
            if t < shape.L - 1:
                np.testing.assert_array_equal(o.h, r.h)
        assert np.all(o.len == 0)
        assert np.all(o.h.astype(np.float16).astype(np.float64) == o.h)
        ulp = np.maximum(np.abs(r.h) * 2.0 ** -10, 2.0 ** -24)
        assert np.all(np.abs(o.h - r.h) <= ulp * (1 + 1e-9))
        mean += o.h
    exact = r.h
    step = np.maximum(np.abs(exact) * 2.0 ** -10, 2.0 ** -24)
    assert np.all(np.abs(mean / K - exact) <= 6 * step / np.sqrt(K))
