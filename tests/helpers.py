"""Shared test plumbing: tolerances and numpy <-> torch marshalling."""
from __future__ import annotations

import numpy as np

# Floating-point gate for FP32-state paths.  The pages state only an "rtol
# 1e-4" check against an FP32 reference.  Reading: per element
#   |y - y_ref| / max(|y_ref|, tau)  <= 1e-4,  tau = 1e-2 * rms(y_ref),
# the floor keeping the relative measure meaningful for outputs that cross
# zero.  Checkpoints use the same rule with the state's rms.
RTOL = 1e-4
FLOOR = 1e-2

# The conventional (in-place) comparison paths of both layer types rewrite
# their FP32 state in place every token, so their own rounding (about 2^-24 of
# the state per step) accumulates like a random walk over the steps since the
# exact start state: after t steps about sqrt(t) * 6e-8 of the state, i.e.
# sqrt(t) * 6e-6 of the floor.  Over up to 1024 steps that is ~2e-4; the gate
# for those paths is 5e-4.  Every replay path (Mamba-2 and Gated DeltaNet
# decode, fold, verify, rollback) rounds its checkpoint only at flushes and
# takes RTOL.
RTOL_INPLACE = 5e-4


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tau = FLOOR * np.sqrt(np.mean(ref * ref))
    if tau == 0:
        tau = 1e-30
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), tau)))


def assert_close(got, ref, what="", rtol=RTOL):
    e = rel_err(got, ref)
    assert e <= rtol, f"{what}: max rel err {e:.3e} > {rtol:.1e}"
    return e


def to_dev(a, dtype=None, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def io_dtype(bf16: bool):
    import torch
    return torch.bfloat16 if bf16 else torch.float32
