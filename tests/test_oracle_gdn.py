"""Pins of the stepwise gated-delta-rule oracle."""
import numpy as np
import pytest

from oracle.gdn import GDNStepwise


def _rand(rng, b=2, H=3, dk=5, dv=4, T=10):
    S0 = rng.standard_normal((b, H, dv, dk)) * 0.3
    q = rng.standard_normal((T, b, H, dk))
    k = rng.standard_normal((T, b, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, b, H, dv))
    alpha = np.exp(-np.logaddexp(0, rng.standard_normal((T, b, H))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, b, H))))
    return S0, q, k, v, alpha, beta


def test_scalar_hand_example():
    """dk = dv = 1: s1 = 0.5*(2 - 0.5*1*1*2) + 0.5*4*1 = 2.5, o1 = 2.5*3 = 7.5."""
    m = GDNStepwise(np.full((1, 1, 1, 1), 2.0))
    o = m.step(np.full((1, 1, 1), 3.0), np.ones((1, 1, 1)), np.full((1, 1, 1), 4.0),
               np.full((1, 1), 0.5), np.full((1, 1), 0.5))
    assert m.S[0, 0, 0, 0] == pytest.approx(2.5, abs=1e-15)
    assert o[0, 0, 0] == pytest.approx(7.5, abs=1e-15)


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(11)
    S0, q, k, v, alpha, _ = _rand(rng)
    m = GDNStepwise(S0)
    prod = np.ones(alpha.shape[1:])
    for t in range(q.shape[0]):
        o = m.step(q[t], k[t], v[t], alpha[t], np.zeros_like(alpha[t]))
        prod = prod * alpha[t]
        want = prod[..., None] * np.einsum("bhvk,bhk->bhv", S0, q[t])
        np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-14)


def test_orthonormal_keys_replace_columns():
    """alpha = beta = 1 and k = e_j: the step writes v into column j and leaves
    every other column as it was (the delta rule's exact overwrite)."""
    rng = np.random.default_rng(12)
    dk, dv = 4, 3
    S0 = rng.standard_normal((1, 1, dv, dk))
    m = GDNStepwise(S0)
    want = S0.copy()
    for j in [2, 0, 3]:
        kk = np.zeros((1, 1, dk))
        kk[0, 0, j] = 1.0
        v = rng.standard_normal((1, 1, dv))
        m.step(kk, kk, v, np.ones((1, 1)), np.ones((1, 1)))
        want[0, 0, :, j] = v[0, 0]
        np.testing.assert_array_equal(m.S, want)


def test_dense_brute_force():
    """Explicit matrices: S <- alpha * S @ (I - beta k k^T) + beta v k^T, on a
    rectangular and a square state (a transposed product only shows there)."""
    for dk, dv in [(5, 4), (4, 4)]:
        _dense_case(dk, dv)


def _dense_case(dk, dv):
    rng = np.random.default_rng(13 + dk * 10 + dv)
    S0, q, k, v, alpha, beta = _rand(rng, dk=dk, dv=dv)
    m = GDNStepwise(S0)
    S = S0.copy()
    b, H, dv, dk = S0.shape
    for t in range(q.shape[0]):
        o = m.step(q[t], k[t], v[t], alpha[t], beta[t])
        for bb in range(b):
            for h in range(H):
                kk = k[t, bb, h][:, None]
                M = np.eye(dk) - beta[t, bb, h] * (kk @ kk.T)
                S[bb, h] = alpha[t, bb, h] * S[bb, h] @ M + beta[t, bb, h] * np.outer(v[t, bb, h], kk[:, 0])
                np.testing.assert_allclose(o[bb, h], S[bb, h] @ q[t, bb, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(m.S, S, rtol=1e-12, atol=1e-13)


def test_unrolled_u_chain():
    """o_t from the start state S_c and the tokens 1..t:
    u_t = q_t, u_{j-1} = alpha_j (u_j - beta_j k_j (k_j . u_j)),
    o_t = S_c u_0 + sum_j beta_j v_j (k_j . u_j)."""
    rng = np.random.default_rng(14)
    S0, q, k, v, alpha, beta = _rand(rng, T=8)
    m = GDNStepwise(S0)
    b, H = S0.shape[:2]
    for t in range(q.shape[0]):
        o = m.step(q[t], k[t], v[t], alpha[t], beta[t])
        for bb in range(b):
            for h in range(H):
                u = q[t, bb, h].copy()
                acc = np.zeros(S0.shape[2])
                for j in range(t, -1, -1):
                    d = k[j, bb, h] @ u
                    acc += beta[j, bb, h] * d * v[j, bb, h]
                    u = alpha[j, bb, h] * (u - beta[j, bb, h] * k[j, bb, h] * d)
                np.testing.assert_allclose(o[bb, h], S0[bb, h] @ u + acc, rtol=1e-11, atol=1e-12)


def _draft_batch(rng, b=3, H=2, dk=6, dv=5, T=4):
    S0, q, k, v, alpha, beta = _rand(rng, b=b, H=H, dk=dk, dv=dv, T=T)
    # [T, b, ...] -> [b, T, ...]
    sw = lambda a: np.swapaxes(a, 0, 1)  # noqa: E731
    return S0, sw(q), sw(k), sw(v), sw(alpha), sw(beta)


def test_verify_equals_sequential_steps_and_commits_nothing():
    """Draft i's output is the output of decoding drafts 1..i one by one; the
    oracle's state is untouched until accept."""
    rng = np.random.default_rng(31)
    S0, q, k, v, alpha, beta = _draft_batch(rng)
    m = GDNStepwise(S0)
    o, states = m.verify(q, k, v, alpha, beta)
    np.testing.assert_array_equal(m.S, S0)
    ref = GDNStepwise(S0)
    for i in range(q.shape[1]):
        oi = ref.step(q[:, i], k[:, i], v[:, i], alpha[:, i], beta[:, i])
        np.testing.assert_allclose(o[:, i], oi, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(states[i], ref.S, rtol=1e-13, atol=1e-14)


def test_verify_accept_prefix_matches_dense_products():
    """Accepting a drafts leaves S_0 (prod_i A_i) + (written terms) of exactly
    those a drafts, built here from dense (I - beta k k^T) products; a = 0
    keeps the state."""
    rng = np.random.default_rng(32)
    S0, q, k, v, alpha, beta = _draft_batch(rng, b=4, T=3)
    m = GDNStepwise(S0)
    _, states = m.verify(q, k, v, alpha, beta)
    accepted = np.array([0, 1, 3, 2])
    m.accept(states, accepted)
    for b, a in enumerate(accepted):
        for h in range(S0.shape[1]):
            S = S0[b, h].copy()
            for i in range(a):
                kk = k[b, i, h][:, None]
                M = np.eye(S.shape[1]) - beta[b, i, h] * (kk @ kk.T)
                S = alpha[b, i, h] * S @ M + beta[b, i, h] * v[b, i, h][:, None] @ kk.T
            np.testing.assert_allclose(m.S[b, h], S, rtol=1e-12, atol=1e-13)


def test_verify_single_draft_is_step():
    rng = np.random.default_rng(33)
    S0, q, k, v, alpha, beta = _draft_batch(rng, T=1)
    a, b_ = GDNStepwise(S0), GDNStepwise(S0)
    o, states = a.verify(q, k, v, alpha, beta)
    a.accept(states, np.ones(S0.shape[0], int))
    ob = b_.step(q[:, 0], k[:, 0], v[:, 0], alpha[:, 0], beta[:, 0])
    np.testing.assert_array_equal(o[:, 0], ob)
    np.testing.assert_array_equal(a.S, b_.S)
