"""Pins of the stepwise Mamba-2 oracle against things other than itself.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, a wrong group index, a decay applied after
instead of before the input term) fails at least one of them.
"""
import math

import numpy as np
import pytest

from oracle.mamba2 import Mamba2Stepwise


def _rand_problem(rng, b=2, H=4, P=3, N=5, G=2, T=20):
    A = -np.exp(rng.uniform(0.0, math.log(16.0), H))
    D = rng.standard_normal(H)
    h0 = rng.standard_normal((b, H, P, N)) * 0.3
    dt = rng.uniform(1e-3, 0.1, (T, b, H))
    x = rng.standard_normal((T, b, H, P))
    B = rng.standard_normal((T, b, G, N)) / math.sqrt(N)
    C = rng.standard_normal((T, b, G, N)) / math.sqrt(N)
    return A, D, h0, dt, x, B, C


def test_scalar_hand_example():
    """H = P = N = G = 1, two tokens worked by hand.

    dt*A = -ln 2 then -2 ln 2, so the decays are 1/2 and 1/4:
      h1 = 0.5*1 + 0.1*1*2 = 0.7        y1 = 0.7*3 + 0.5*1 = 2.6
      h2 = 0.25*0.7 + 0.2*(-2)*1 = -0.225  y2 = -0.225*(-1) + 0.5*(-2) = -0.775
    """
    A = np.array([-10.0 * math.log(2.0)])
    D = np.array([0.5])
    m = Mamba2Stepwise(A, D, 1, np.ones((1, 1, 1, 1)))
    y1 = m.step(np.array([[0.1]]), np.array([[[1.0]]]), np.array([[[2.0]]]), np.array([[[3.0]]]))
    assert y1[0, 0, 0] == pytest.approx(2.6, abs=1e-14)
    assert m.h[0, 0, 0, 0] == pytest.approx(0.7, abs=1e-14)
    y2 = m.step(np.array([[0.2]]), np.array([[[-2.0]]]), np.array([[[1.0]]]), np.array([[[-1.0]]]))
    assert m.h[0, 0, 0, 0] == pytest.approx(-0.225, abs=1e-14)
    assert y2[0, 0, 0] == pytest.approx(-0.775, abs=1e-14)


def test_no_decay_is_cumulative_sum():
    """A = 0: the state is h0 plus the running sum of dt x B^T (numpy cumsum)."""
    rng = np.random.default_rng(1)
    _, D, h0, dt, x, B, C = _rand_problem(rng)
    H, G = h0.shape[1], B.shape[2]
    g = np.arange(H) // (H // G)
    m = Mamba2Stepwise(np.zeros(H), D, G, h0)
    inc = dt[..., None, None] * x[..., None] * B[:, :, g, None, :]     # [T,b,H,P,N]
    states = h0[None] + np.cumsum(inc, axis=0)
    for t in range(dt.shape[0]):
        y = m.step(dt[t], x[t], B[t], C[t])
        want = np.einsum("bhpn,bhn->bhp", states[t], C[t][:, g]) + D[None, :, None] * x[t]
        np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(m.h, states[t], rtol=1e-12, atol=1e-12)


def test_vanishing_dt_reads_checkpoint():
    """dt -> 0: no decay, no input; y = h0 C + D x."""
    rng = np.random.default_rng(2)
    A, D, h0, dt, x, B, C = _rand_problem(rng, T=3)
    H, G = h0.shape[1], B.shape[2]
    g = np.arange(H) // (H // G)
    m = Mamba2Stepwise(A, D, G, h0)
    for t in range(3):
        y = m.step(np.full_like(dt[t], 1e-13), x[t], B[t], C[t])
        want = np.einsum("bhpn,bhn->bhp", h0, C[t][:, g]) + D[None, :, None] * x[t]
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-10)


def _brute_unrolled(A, D, h0, dt, x, B, C):
    """Independent O(T^2) loops over the unrolled sum, decays as products of
    per-token factors; group of head h computed as (h*G)//H."""
    T, b, H = dt.shape
    P, N, G = h0.shape[2], h0.shape[3], B.shape[2]
    out = np.zeros((T, b, H, P))
    for bb in range(b):
        for h in range(H):
            g = (h * G) // H
            for t in range(T):
                decay0 = 1.0
                for i in range(t + 1):
                    decay0 *= math.exp(dt[i, bb, h] * A[h])
                for p in range(P):
                    acc = decay0 * sum(h0[bb, h, p, n] * C[t, bb, g, n] for n in range(N))
                    for j in range(t + 1):
                        w = dt[j, bb, h]
                        for i in range(j + 1, t + 1):
                            w *= math.exp(dt[i, bb, h] * A[h])
                        cb = sum(B[j, bb, g, n] * C[t, bb, g, n] for n in range(N))
                        acc += w * cb * x[j, bb, h, p]
                    out[t, bb, h, p] = acc + D[h] * x[t, bb, h, p]
    return out


def test_brute_force_unrolled_sum():
    rng = np.random.default_rng(3)
    A, D, h0, dt, x, B, C = _rand_problem(rng, b=2, H=4, P=3, N=5, G=2, T=12)
    want = _brute_unrolled(A, D, h0, dt, x, B, C)
    m = Mamba2Stepwise(A, D, 2, h0)
    for t in range(dt.shape[0]):
        np.testing.assert_allclose(m.step(dt[t], x[t], B[t], C[t]), want[t], rtol=1e-11, atol=1e-12)


def test_semiseparable_matrix_form():
    """From a zero state, Y = (M o (C B^T)) X with M[t,j] = exp(A (S_t - S_j)) dt_j
    for j <= t (S = cumulative dt): the materialised matrix form of a selective
    SSM, evaluated with one matrix product per head."""
    rng = np.random.default_rng(4)
    A, D, _, dt, x, B, C = _rand_problem(rng, b=1, H=2, P=4, N=6, G=1, T=16)
    T = dt.shape[0]
    m = Mamba2Stepwise(A, D, 1, np.zeros((1, 2, 4, 6)))
    ys = np.stack([m.step(dt[t], x[t], B[t], C[t]) for t in range(T)])   # [T,1,H,P]
    for h in range(2):
        S = np.cumsum(dt[:, 0, h])
        mask = np.tril(np.exp(A[h] * (S[:, None] - S[None, :])) * dt[None, :, 0, h])
        CB = C[:, 0, 0, :] @ B[:, 0, 0, :].T                              # [T,T]
        Y = (mask * CB) @ x[:, 0, h, :] + D[h] * x[:, 0, h, :]
        np.testing.assert_allclose(ys[:, 0, h, :], Y, rtol=1e-11, atol=1e-12)


def test_groups_are_separate():
    """Changing group 1's B and C leaves the heads of group 0 untouched."""
    rng = np.random.default_rng(5)
    A, D, h0, dt, x, B, C = _rand_problem(rng, b=1, H=4, P=2, N=3, G=2, T=4)
    m1, m2 = Mamba2Stepwise(A, D, 2, h0), Mamba2Stepwise(A, D, 2, h0)
    B2, C2 = B.copy(), C.copy()
    B2[:, :, 1] += 1.0
    C2[:, :, 1] -= 0.5
    for t in range(4):
        y1 = m1.step(dt[t], x[t], B[t], C[t])
        y2 = m2.step(dt[t], x[t], B2[t], C2[t])
        np.testing.assert_array_equal(y1[:, :2], y2[:, :2])
        assert np.all(np.abs(y1[:, 2:] - y2[:, 2:]) > 0)


def test_linear_in_state_and_input():
    """With dt fixed, y is linear in (h0, x) jointly."""
    rng = np.random.default_rng(6)
    A, D, h0, dt, x, B, C = _rand_problem(rng, T=5)
    m1, m2 = Mamba2Stepwise(A, D, 2, h0), Mamba2Stepwise(A, D, 2, 2.5 * h0)
    for t in range(5):
        np.testing.assert_allclose(m2.step(dt[t], 2.5 * x[t], B[t], C[t]),
                                   2.5 * m1.step(dt[t], x[t], B[t], C[t]), rtol=1e-12, atol=1e-13)


def test_verify_and_accept_equal_stepwise_prefix():
    """Scoring T drafts equals decoding them one by one; accepting a of them
    leaves the state of decoding exactly those a."""
    rng = np.random.default_rng(7)
    A, D, h0, dt, x, B, C = _rand_problem(rng, b=3, T=4)
    dtd, xd, Bd, Cd = (np.moveaxis(a, 0, 1) for a in (dt, x, B, C))   # [b,T,...]
    m = Mamba2Stepwise(A, D, 2, h0)
    y, states = m.verify(dtd, xd, Bd, Cd)
    ref = Mamba2Stepwise(A, D, 2, h0)
    for t in range(4):
        np.testing.assert_array_equal(y[:, t], ref.step(dt[t], x[t], B[t], C[t]))
    np.testing.assert_array_equal(m.h, h0)          # nothing committed
    acc = np.array([0, 2, 4])
    m.accept(states, acc)
    for bb, a in enumerate(acc):
        r = Mamba2Stepwise(A, D, 2, h0[bb:bb + 1])
        for t in range(a):
            r.step(dt[t, bb:bb + 1], x[t, bb:bb + 1], B[t, bb:bb + 1], C[t, bb:bb + 1])
        np.testing.assert_array_equal(m.h[bb], r.h[0])
