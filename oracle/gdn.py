"""Stepwise gated delta rule (Gated DeltaNet decode), float64 -- the oracle.

TEST INFRASTRUCTURE (see the package docstring): never imported by the product.

Gated DeltaNet is one of the two SSM layer types the method ships kernels for
([AT Pulse] §Capabilities and access, layer types).  The pages print no
equation for it; the recurrence used is the one of the Gated DeltaNet decode
workload (state S is dv x dk per head):

    S <- alpha * S (I - beta k k^T) + beta v k^T
    o <- S q

written here in its rank-one form  S - beta (S k) k^T  (the dense product with
(I - beta k k^T) is the brute-force pin in the tests).  Reading: no 1/sqrt(dk)
output scale; q and k are used exactly as given (already L2-normalised and
rounded by the input generator).
"""
from __future__ import annotations

import numpy as np


class GDNStepwise:
    """Batched stepwise gated delta rule.  State ``S`` is [b, H, dv, dk] float64."""

    def __init__(self, S0):
        self.S = np.array(S0, dtype=np.float64, copy=True)

    def _update(self, S, q, k, v, alpha, beta):
        q = np.asarray(q, np.float64)          # [b, H, dk]
        k = np.asarray(k, np.float64)          # [b, H, dk]
        v = np.asarray(v, np.float64)          # [b, H, dv]
        alpha = np.asarray(alpha, np.float64)[:, :, None, None]
        beta = np.asarray(beta, np.float64)[:, :, None, None]
        Sk = np.einsum("bhvk,bhk->bhv", S, k)                   # S k
        S = alpha * (S - beta * Sk[..., None] * k[:, :, None, :]) \
            + beta * v[..., None] * k[:, :, None, :]
        o = np.einsum("bhvk,bhk->bhv", S, q)
        return S, o

    def step(self, q, k, v, alpha, beta) -> np.ndarray:
        """One decode token for every sequence; returns o [b, H, dv]."""
        self.S, o = self._update(self.S, q, k, v, alpha, beta)
        return o

    def verify(self, q, k, v, alpha, beta):
        """Score T draft tokens per sequence (inputs [b, T, H, ...]) without
        committing: draft i is decoded on top of drafts 1..i, as speculative
        decoding scores them (AT Pulse, Technical analysis: output-only
        evaluation of the drafts; rollback keeps the accepted prefix).

        Returns (o [b, T, H, dv], states) where states[i] is the state after
        drafts 1..i+1; ``accept`` keeps one of them per sequence."""
        T = np.asarray(alpha).shape[1]
        S = self.S
        outs, states = [], []
        for i in range(T):
            S, o = self._update(S, q[:, i], k[:, i], v[:, i], alpha[:, i], beta[:, i])
            outs.append(o)
            states.append(S)
        return np.stack(outs, axis=1), states

    def accept(self, states, accepted) -> None:
        """Keep, per sequence, the state after its accepted prefix (0 = unchanged)."""
        new = self.S.copy()
        for b, a in enumerate(np.asarray(accepted)):
            if a > 0:
                new[b] = states[a - 1][b]
        self.S = new
