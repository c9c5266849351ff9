"""CPU checks of two identities the Gated DeltaNet fold kernels rely on.

1. The re-associated fold.  Folding nrec records into a state row-wise with the
   records' Gram matrix -- p_j = s . k_j, C_ij = (k_i . k_j) prod_{i<m<j} alpha_m,
   a_j / g_j / A the prefix / suffix / total products of alpha, d_j = a_j p_j +
   sum_{i<j} C_ij e_i, e_j = beta_j (v_j[r] - alpha_j d_j), new row A s +
   sum_j e_j g_j k_j -- equals the oracle's sequential gated delta steps
   S <- alpha S (I - beta k k^T) + beta v k^T, oldest record first.  Both the
   CUDA-core fold and the tensor-core fold phase compute this form; here it is
   written out in float64 from those definitions and compared with
   oracle.gdn.GDNStepwise.

2. The three-term bf16 split.  Every float32 x = 0 or with 2^-110 <= |x| <= the
   largest finite bf16 is exactly t1 + t2 + t3 with t1 the nearest bf16 to x, t2
   the nearest to x - t1 and t3 = x - t1 - t2 a bf16 itself: the tensor-core
   fold's products of split factors with bf16 keys are then exact.  Round to
   nearest even to bf16 is emulated on the bits.
"""
import numpy as np
import pytest

from oracle.gdn import GDNStepwise


def _fold_reassociated(S, K, V, al, be):
    """S [dv, dk], K [n, dk], V [n, dv], al / be [n] -> folded state (float64)."""
    n = K.shape[0]
    P = S @ K.T                                         # [dv, n]: p_j of every row
    G = K @ K.T
    a = np.array([np.prod(al[:j]) for j in range(n)])
    g = np.array([np.prod(al[j + 1:]) for j in range(n)])
    A = np.prod(al)
    C = np.zeros((n, n))
    for i in range(n):
        for j in range(i + 1, n):
            C[i, j] = G[i, j] * np.prod(al[i + 1:j])
    E = np.zeros_like(P)                                # e_j of every row
    for j in range(n):
        d = a[j] * P[:, j] + E[:, :j] @ C[:j, j]
        E[:, j] = be[j] * (V[j] - al[j] * d)
    return A * S + (E * g[None, :]) @ K


@pytest.mark.parametrize("n", [1, 2, 3, 8, 16, 17])
def test_reassociated_fold_equals_sequential_steps(n):
    rng = np.random.default_rng(100 + n)
    dk, dv = 32, 24
    S0 = rng.standard_normal((dv, dk)) * 0.1
    K = rng.standard_normal((n, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = rng.standard_normal((n, dv))
    al = np.exp(-np.log1p(np.exp(rng.standard_normal(n))))   # exp(-softplus), the input recipe's alpha
    be = 1.0 / (1.0 + np.exp(-rng.standard_normal(n)))
    orc = GDNStepwise(S0[None, None])
    q = np.zeros((1, 1, dk))
    for j in range(n):
        orc.step(q, K[j][None, None], V[j][None, None], al[j:j + 1][None], be[j:j + 1][None])
    got = _fold_reassociated(S0, K, V, al, be)
    ref = orc.S[0, 0]
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_reassociated_fold_catches_a_dropped_term():
    # the check above is not vacuous: leaving out the Gram coupling changes the result
    rng = np.random.default_rng(7)
    n, dk, dv = 6, 16, 8
    S0 = rng.standard_normal((dv, dk)) * 0.1
    K = rng.standard_normal((n, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V, al, be = rng.standard_normal((n, dv)), np.full(n, 0.9), np.full(n, 0.5)
    orc = GDNStepwise(S0[None, None])
    for j in range(n):
        orc.step(np.zeros((1, 1, dk)), K[j][None, None], V[j][None, None], al[j:j + 1][None], be[j:j + 1][None])
    P = S0 @ K.T
    E = np.stack([be[j] * (V[j] - al[j] * np.prod(al[:j]) * P[:, j]) for j in range(n)], axis=1)
    g = np.array([np.prod(al[j + 1:]) for j in range(n)])
    no_gram = np.prod(al) * S0 + (E * g[None, :]) @ K
    assert np.max(np.abs(no_gram - orc.S[0, 0])) > 1e-3


def _bf16_rn(x):
    """float32 array -> nearest bf16 (ties to even), as float32."""
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def test_three_term_bf16_split_is_exact():
    rng = np.random.default_rng(3)
    bf16_max = np.array([0x7F7F0000], dtype=np.uint32).view(np.float32)[0]     # ~3.39e38
    mant = rng.uniform(1.0, 2.0, 200_000)
    expo = rng.integers(-110, 127, mant.size)
    x = (mant * np.exp2(expo) * rng.choice([-1.0, 1.0], mant.size)).astype(np.float32)
    x = x[np.abs(x) <= bf16_max]
    x = np.concatenate([x, np.array([1.0, -1.0, 0.0, 2.0 ** -110, -(2.0 ** -110), bf16_max, -bf16_max,
                                     np.nextafter(np.float32(1), np.float32(2)), 1.9999999], dtype=np.float32)])
    t1 = _bf16_rn(x)
    r1 = (x - t1).astype(np.float32)                    # exact (Sterbenz)
    assert np.array_equal(r1.astype(np.float64), x.astype(np.float64) - t1.astype(np.float64))
    t2 = _bf16_rn(r1)
    r2 = (r1 - t2).astype(np.float32)
    t3 = _bf16_rn(r2)
    assert np.array_equal(t3, r2)                       # what is left is a bf16 itself
    total = t1.astype(np.float64) + t2.astype(np.float64) + t3.astype(np.float64)
    assert np.array_equal(total, x.astype(np.float64))
