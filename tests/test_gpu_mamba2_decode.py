"""Replay decode (with fused flush) and the conventional decode against the oracle."""
import numpy as np
import pytest

from ssm_decode_state_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def _run(shape, seed, steps, h0=None, sample=None, prefill=0, first_step=1000, **kw):
    from tests.m2_runner import M2Run
    r = M2Run(shape, seed, h0=h0, sample=sample, **kw)
    if prefill:
        r.prefill_conventional(range(prefill))
    flushes = 0
    for t in range(steps):
        _, _, folded = r.decode(first_step + t)
        flushes += folded[r.sample[0]] is not None
        if t % 7 == 0:
            r.check_records(seqs=list(r.sample))
    return r, flushes


def test_tiny_fp32_every_step():
    """Tiny Mamba-2 layer, FP32 throughout: 32-token stepwise prefill, then 64
    decode steps compared at every step, including the 4 flushes."""
    w = gen.workloads()["mamba2_tiny"]
    r, flushes = _run(w.shape, w.seed, w.steps, prefill=w.prefill)
    assert flushes == 4
    print("tiny max errors", r.max_err)


@pytest.mark.parametrize("L", [1, 4, 16])
def test_ragged_multi_tile(L):
    """Two CTAs per head (rows split 24 + 24), a headdim that is not a power
    of two, two groups, bf16 inputs."""
    shape = gen.Mamba2Shape(batch=3, nheads=8, headdim=48, dstate=32, ngroups=2, L=L)
    h0 = gen.mamba2_random_state(shape, 77)
    r, flushes = _run(shape, 77, 37, h0=h0)
    assert flushes == (37 // L)


@pytest.mark.parametrize("N,P", [(16, 64), (64, 32), (128, 256)])
def test_dstate_headdim_variants(N, P):
    shape = gen.Mamba2Shape(batch=2, nheads=4, headdim=P, dstate=N, ngroups=2, L=8)
    h0 = gen.mamba2_random_state(shape, 5)
    _run(shape, 5, 20, h0=h0)


def test_batch_one_serving_shape():
    """Batch 1 at the serving head shape: the persistent kernel with one head per
    work item and fewer CTAs than SMs."""
    shape = gen.Mamba2Shape(batch=1, nheads=128, headdim=64, dstate=128, ngroups=8, L=16)
    h0 = gen.mamba2_random_state(shape, 9)
    _run(shape, 9, 34, h0=h0)


def test_batch_one_split_rows():
    """Batch 1 at a shape the per-tile kernel serves (headdim 128, dstate 64):
    the rows of a head are split over several CTAs to fill the GPU."""
    shape = gen.Mamba2Shape(batch=1, nheads=16, headdim=128, dstate=64, ngroups=4, L=8)
    h0 = gen.mamba2_random_state(shape, 19)
    _run(shape, 19, 20, h0=h0)


def test_serving_shape_b256_sampled():
    """Mamba-2 layer at serving shape (nheads 128, headdim 64, dstate 128,
    ngroups 8, 4 MiB state per sequence), batch 256, 256 decode steps from a
    random N(0, 0.1) state; the oracle follows 3 sequences, ring pointers are
    checked for all 256 at every step."""
    w = gen.workloads()["mamba2_b256"]
    sample = [0, 131, 255]
    h0 = gen.mamba2_random_state(w.shape, w.seed)
    r, flushes = _run(w.shape, w.seed, w.steps, h0=h0, sample=sample)
    assert flushes == w.steps // 16
    print("b256 max errors", r.max_err)


def test_run_twice_bitwise():
    shape = gen.Mamba2Shape(batch=4, nheads=8, headdim=32, dstate=64, ngroups=2, L=4)
    h0 = gen.mamba2_random_state(shape, 3)
    outs = []
    for _ in range(2):
        r, _ = _run(shape, 3, 9, h0=h0)
        outs.append((r.cache.ckpt.cpu().numpy(), r.cache.rec_x.float().cpu().numpy()))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
