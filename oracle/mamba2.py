"""Stepwise Mamba-2 SSM decode recurrence, float64 -- the oracle.

TEST INFRASTRUCTURE (see the package docstring): never imported by the product.

What it computes.  Per sequence b and head h, with g(h) the group of head h,
one decode token (dt, x, B, C) updates the (headdim x dstate) state and reads
the output from it:

    h <- exp(dt * A_h) * h + dt * outer(x, B_g(h))
    y <- h @ C_g(h) + D_h * x

This is the conventional decode step that "updates the state, reads the
output from it, and stores it" ([Clarity] claim ledger [6]); the replay
method reaches exactly this result, re-associated, from a checkpoint plus the
buffered records ([AT Pulse] §Technical analysis, core idea: the recurrence
unrolled over a window of L tokens; [Clarity] claim ledger [17], [18]).  So
the oracle is the stepwise definition itself.

Readings where the pages are silent (they print no equation):

* discretisation: exp(dt*A) decay and dt*B input scaling (the Mamba-2
  zero-order-hold A / Euler B form); dt arrives already positive;
* A and D are per head; heads map to groups contiguously,
  g(h) = floor(h / (nheads / ngroups));
* speculative verify scores draft i causally (it sees the accepted past plus
  drafts 1..i) and does not commit; accepting a prefix of a drafts leaves the
  state exactly as if those a tokens had been decoded and the rest never
  seen ([AT Pulse] §Technical analysis, speculative decoding: rollback as a
  buffer-pointer move; [Clarity] claim ledger [12], [13]).
"""
from __future__ import annotations

import numpy as np


def group_of_head(nheads: int, ngroups: int) -> np.ndarray:
    return np.arange(nheads) // (nheads // ngroups)


class Mamba2Stepwise:
    """Batched stepwise recurrence.  State ``h`` is [b, H, P, N] float64."""

    def __init__(self, A, D, ngroups: int, h0):
        self.A = np.asarray(A, np.float64)
        self.D = np.asarray(D, np.float64)
        self.h = np.array(h0, dtype=np.float64, copy=True)
        self.g = group_of_head(self.A.shape[0], ngroups)

    # one token for every sequence of the batch
    def _update(self, h, dt, x, B, C):
        dt = np.asarray(dt, np.float64)                 # [b, H]
        x = np.asarray(x, np.float64)                   # [b, H, P]
        Bh = np.asarray(B, np.float64)[:, self.g, :]    # [b, H, N]
        Ch = np.asarray(C, np.float64)[:, self.g, :]    # [b, H, N]
        a = np.exp(dt * self.A[None, :])                # per-step decay exp(dt*A)
        h = a[:, :, None, None] * h + (dt[:, :, None] * x)[:, :, :, None] * Bh[:, :, None, :]
        y = np.einsum("bhpn,bhn->bhp", h, Ch) + self.D[None, :, None] * x
        return h, y

    def step(self, dt, x, B, C) -> np.ndarray:
        """Decode one token: update the state and return y [b, H, P]."""
        self.h, y = self._update(self.h, dt, x, B, C)
        return y

    def verify(self, dt, x, B, C):
        """Score T drafts per sequence (inputs [b, T, ...]) without committing.

        Returns (y [b, T, H, P], states) where states[i] is the state after
        drafts 1..i+1; ``accept`` picks one of them per sequence."""
        T = dt.shape[1]
        h = self.h
        ys, states = [], []
        for i in range(T):
            h, y = self._update(h, dt[:, i], x[:, i], B[:, i], C[:, i])
            ys.append(y)
            states.append(h)
        return np.stack(ys, axis=1), states

    def accept(self, states, accepted) -> None:
        """Keep, per sequence, the state after its accepted prefix (0 = unchanged)."""
        accepted = np.asarray(accepted)
        new = self.h.copy()
        for b, a in enumerate(accepted):
            if a > 0:
                new[b] = states[a - 1][b]
        self.h = new
