"""Seeded synthetic inputs for the ReplaySSM decode workloads.

This module only draws random numbers with the shapes and value distributions
of the workloads; it holds none of the method's arithmetic.  Both the CUDA path
(through the tests and the bench) and the CPU oracle consume what it returns.

Every array comes from numpy's PCG64 generator seeded with ``(seed, stream,
index)``, so the same call gives the same bits on x86 and Arm hosts.  Values
that the kernels read as bf16 are rounded to bf16 here (round to nearest even)
and returned as float32 arrays that hold exactly those bf16 values, so the
oracle widens the very numbers the GPU sees.

Distributions (the workload descriptions of the Mamba-2 and Gated DeltaNet
decode configurations):

* Mamba-2: x ~ N(0,1); B, C ~ N(0,1)/sqrt(dstate);
  dt = clamp(softplus(N(0,1) + bias_h), 1e-3, 0.1), with a per-head bias
  bias_h = softplus^-1(dt0_h) and dt0_h log-uniform in [1e-3, 0.1];
  A_h = -exp(U(log 1, log 16)); D_h ~ N(0,1); a random initial state has
  entries ~ N(0, 0.1^2) (std 0.1).
* Gated DeltaNet: q, k ~ N(0,1) then L2-normalised in float32 and rounded to
  bf16; v ~ N(0,1) in bf16; alpha = exp(-softplus(N(0,1))); beta =
  sigmoid(N(0,1)); initial state entries ~ N(0, 0.1^2).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_STREAM_PARAMS = 1
_STREAM_STATE = 2
_STREAM_STEP = 3
_STREAM_DRAFT = 4
_STREAM_ACCEPT = 5


def _rng(seed: int, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, index])))


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), kept as float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    nan = np.isnan(a)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    out = r.view(np.float32).copy()
    out[nan] = np.nan
    return out


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-representable."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, z)


# --------------------------------------------------------------------------
# Mamba-2
# --------------------------------------------------------------------------

@dataclass
class Mamba2Shape:
    batch: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    L: int = 16
    bf16_io: bool = True          # x, B, C (and their records) in bf16; else fp32

    def group_of_head(self) -> np.ndarray:
        """g(h) = floor(h / (nheads / ngroups)): contiguous heads share a group."""
        return np.arange(self.nheads) // (self.nheads // self.ngroups)


@dataclass
class Mamba2Params:
    A: np.ndarray        # [H] float32, negative
    D: np.ndarray        # [H] float32
    dt_bias: np.ndarray  # [H] float32


@dataclass
class Mamba2Step:
    dt: np.ndarray  # [b, H] float32 (or [b, T, H] for drafts)
    x: np.ndarray   # [b, H, P]      (or [b, T, H, P])
    B: np.ndarray   # [b, G, N]      (or [b, T, G, N])
    C: np.ndarray   # [b, G, N]      (or [b, T, G, N])


def mamba2_params(shape: Mamba2Shape, seed: int) -> Mamba2Params:
    r = _rng(seed, _STREAM_PARAMS)
    H = shape.nheads
    A = -np.exp(r.uniform(np.log(1.0), np.log(16.0), size=H))
    D = r.standard_normal(H)
    dt0 = np.exp(r.uniform(np.log(1e-3), np.log(0.1), size=H))
    bias = np.log(np.expm1(dt0))                       # softplus^-1(dt0)
    return Mamba2Params(A=A.astype(np.float32), D=D.astype(np.float32),
                        dt_bias=bias.astype(np.float32))


def mamba2_random_state(shape: Mamba2Shape, seed: int, std: float = 0.1,
                        batch_slice: slice | None = None) -> np.ndarray:
    """[b, H, P, N] float32 with entries ~ N(0, std^2); each sequence has its own
    stream, so a slice of sequences can be drawn without drawing the rest."""
    bs = range(shape.batch)[batch_slice] if batch_slice is not None else range(shape.batch)
    out = np.empty((len(bs), shape.nheads, shape.headdim, shape.dstate), np.float32)
    for i, b in enumerate(bs):
        r = _rng(seed, _STREAM_STATE, b)
        out[i] = r.standard_normal((shape.nheads, shape.headdim, shape.dstate),
                                   dtype=np.float32)
        out[i] *= np.float32(std)
    return out


def _mamba2_tokens(shape: Mamba2Shape, params: Mamba2Params, r: np.random.Generator,
                   lead: tuple) -> Mamba2Step:
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    z = r.standard_normal(lead + (H,))
    dt = np.clip(_softplus(z + params.dt_bias.astype(np.float64)), 1e-3, 0.1).astype(np.float32)
    x = r.standard_normal(lead + (H, P), dtype=np.float32)
    Bm = (r.standard_normal(lead + (G, N)) / np.sqrt(N)).astype(np.float32)
    Cm = (r.standard_normal(lead + (G, N)) / np.sqrt(N)).astype(np.float32)
    if shape.bf16_io:
        x, Bm, Cm = round_bf16(x), round_bf16(Bm), round_bf16(Cm)
    return Mamba2Step(dt=dt, x=x, B=Bm, C=Cm)


def mamba2_step_inputs(shape: Mamba2Shape, params: Mamba2Params, seed: int, step: int,
                       batch: int | None = None) -> Mamba2Step:
    """Inputs of decode step ``step`` for all sequences: dt [b,H], x [b,H,P], B/C [b,G,N]."""
    b = shape.batch if batch is None else batch
    return _mamba2_tokens(shape, params, _rng(seed, _STREAM_STEP, step), (b,))


def mamba2_draft_inputs(shape: Mamba2Shape, params: Mamba2Params, seed: int, step: int,
                        T: int) -> Mamba2Step:
    """T draft tokens per sequence: dt [b,T,H], x [b,T,H,P], B/C [b,T,G,N]."""
    return _mamba2_tokens(shape, params, _rng(seed, _STREAM_DRAFT, step), (shape.batch, T))


def accepted_counts(batch: int, T: int, seed: int, step: int) -> np.ndarray:
    """Accepted draft-prefix length per sequence, uniform on {0..T}, int32 [b]."""
    return _rng(seed, _STREAM_ACCEPT, step).integers(0, T + 1, size=batch).astype(np.int32)


# --------------------------------------------------------------------------
# Gated DeltaNet
# --------------------------------------------------------------------------

@dataclass
class GDNShape:
    batch: int
    nheads: int
    dk: int
    dv: int
    L: int = 16


@dataclass
class GDNStep:
    q: np.ndarray      # [b, H, dk] (bf16 values)
    k: np.ndarray      # [b, H, dk] (bf16 values)
    v: np.ndarray      # [b, H, dv] (bf16 values)
    alpha: np.ndarray  # [b, H] float32
    beta: np.ndarray   # [b, H] float32


def gdn_random_state(shape: GDNShape, seed: int, std: float = 0.1,
                     batch_slice: slice | None = None) -> np.ndarray:
    """[b, H, dv, dk] float32, entries ~ N(0, std^2), one stream per sequence."""
    bs = range(shape.batch)[batch_slice] if batch_slice is not None else range(shape.batch)
    out = np.empty((len(bs), shape.nheads, shape.dv, shape.dk), np.float32)
    for i, b in enumerate(bs):
        r = _rng(seed, _STREAM_STATE, b)
        out[i] = r.standard_normal((shape.nheads, shape.dv, shape.dk), dtype=np.float32)
        out[i] *= np.float32(std)
    return out


def _l2norm_f32(a: np.ndarray) -> np.ndarray:
    a = a.astype(np.float32)
    n = np.sqrt(np.sum(a * a, axis=-1, keepdims=True, dtype=np.float32))
    return (a / n).astype(np.float32)


def _gdn_tokens(shape: GDNShape, r, lead: tuple) -> GDNStep:
    H = shape.nheads
    q = round_bf16(_l2norm_f32(r.standard_normal(lead + (H, shape.dk), dtype=np.float32)))
    k = round_bf16(_l2norm_f32(r.standard_normal(lead + (H, shape.dk), dtype=np.float32)))
    v = round_bf16(r.standard_normal(lead + (H, shape.dv), dtype=np.float32))
    alpha = np.exp(-_softplus(r.standard_normal(lead + (H,)))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-r.standard_normal(lead + (H,))))).astype(np.float32)
    return GDNStep(q=q, k=k, v=v, alpha=alpha, beta=beta)


def gdn_step_inputs(shape: GDNShape, seed: int, step: int) -> GDNStep:
    """One token per sequence: q, k [b, H, dk], v [b, H, dv], alpha, beta [b, H]."""
    return _gdn_tokens(shape, _rng(seed, _STREAM_STEP, step), (shape.batch,))


def gdn_draft_inputs(shape: GDNShape, seed: int, step: int, T: int) -> GDNStep:
    """T draft tokens per sequence: q, k [b, T, H, dk], v [b, T, H, dv], alpha, beta [b, T, H]."""
    return _gdn_tokens(shape, _rng(seed, _STREAM_DRAFT, step), (shape.batch, T))


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    kind: str                  # "mamba2" | "mamba2_fp8" | "mamba2_verify" | "gdn" | "gdn_verify"
    shape: object
    steps: int
    seed: int
    prefill: int = 0           # stepwise prefill tokens from a zero state (tiny case)
    T: int = 0                 # drafts per verify step
    extra: dict = field(default_factory=dict)


def workloads() -> dict[str, Workload]:
    return {
        "mamba2_tiny": Workload(
            "mamba2_tiny", "mamba2",
            Mamba2Shape(batch=2, nheads=4, headdim=16, dstate=16, ngroups=1, L=16, bf16_io=False),
            steps=64, seed=1000, prefill=32),
        "mamba2_b256": Workload(
            "mamba2_b256", "mamba2",
            Mamba2Shape(batch=256, nheads=128, headdim=64, dstate=128, ngroups=8, L=16),
            steps=256, seed=1001),
        "mamba2_fp8read_b256": Workload(
            "mamba2_fp8read_b256", "mamba2_fp8",
            Mamba2Shape(batch=256, nheads=128, headdim=64, dstate=128, ngroups=8, L=16),
            steps=1024, seed=1002),
        "mamba2_nvfp4read_b256": Workload(
            "mamba2_nvfp4read_b256", "mamba2_nvfp4",
            Mamba2Shape(batch=256, nheads=128, headdim=64, dstate=128, ngroups=8, L=16),
            steps=1024, seed=1006),
        "mamba2_f16ckpt_b256": Workload(
            "mamba2_f16ckpt_b256", "mamba2_f16ckpt",
            Mamba2Shape(batch=256, nheads=128, headdim=64, dstate=128, ngroups=8, L=16),
            steps=1024, seed=1007),
        "mamba2_verify_b512_T4": Workload(
            "mamba2_verify_b512_T4", "mamba2_verify",
            Mamba2Shape(batch=512, nheads=128, headdim=64, dstate=128, ngroups=8, L=16),
            steps=200, seed=1003, T=4),
        "gdn_b256": Workload(
            "gdn_b256", "gdn",
            GDNShape(batch=256, nheads=32, dk=128, dv=128, L=16),
            steps=256, seed=1004),
        # the first next row: Gated DeltaNet speculative verify of 4 drafts on the
        # batch-256 GDN layer (the verify step of the Mamba-2 verify workload, on GDN)
        "gdn_verify_b256_T4": Workload(
            "gdn_verify_b256_T4", "gdn_verify",
            GDNShape(batch=256, nheads=32, dk=128, dv=128, L=16),
            steps=200, seed=1005, T=4),
    }
