"""The single-pass small-batch replay decode (batches up to 16 of the serving
shape with a float32 checkpoint).

Every sequence of batches 1, 3, 4, 8 and 16 is followed by the oracle over 17
decode steps from staggered rings (each sequence takes one fused flush, ring
runs wrap around the ring end): y at every step, the folded checkpoints, the
appended records and the ring pointers exact, then a standalone flush.  A second
test drives one cache at batch 32 (above the small-batch limit of 16: the
persistent kernel) and a copy of it through slot-mapped calls of 8 or 4
sequences per step (the small-batch kernel): both kernels form every sum in the
same order, so outputs, checkpoints and records must agree bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle.mamba2 import Mamba2Stepwise
from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL, assert_close, rel_err
from tests.test_gpu_full_batch import _check_ring, _dev, _m2_oracle_prefill, _m2_prefill, _ring_model, _stagger

pytestmark = pytest.mark.gpu

FIELDS = ("ckpt", "rec_dt", "rec_x", "rec_B", "rec_C", "ring_head", "ring_len")


def _serving(batch):
    w = gen.workloads()["mamba2_b256"]
    s = w.shape
    return gen.Mamba2Shape(batch, s.nheads, s.headdim, s.dstate, s.ngroups, s.L, True), w.seed


@pytest.mark.parametrize("batch", [1, 3, 4, 8, 16])
def test_small_batch_every_sequence(batch):
    from ssm_decode_state_gb300 import replayssm as rs
    shape, seed = _serving(batch)
    seed += batch
    prm = gen.mamba2_params(shape, seed)
    h0 = gen.mamba2_random_state(shape, seed)
    dims = rs.mamba2_dims(batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D),
                            ckpt=torch.from_numpy(h0).cuda())
    lens, heads = _stagger(batch, shape.L, shape.L - 1)
    pre = _m2_prefill(cache, shape, prm, seed, lens, heads)
    ring = _ring_model(lens, heads, shape.L)
    orc = Mamba2Stepwise(prm.A, prm.D, shape.ngroups, h0)
    _m2_oracle_prefill(orc, pre, lens, np.arange(batch))
    folded_seqs = set()
    for t in range(shape.L + 1):
        st = gen.mamba2_step_inputs(shape, prm, seed, t)
        slot = np.array([(s.head + s.len) % shape.L for s in ring.seqs])
        y = rs.decode(cache, *_dev(st))
        folded = np.array([f is not None for f in ring.decode([t] * batch)])
        _check_ring(cache, ring)
        yo = orc.step(st.dt, st.x, st.B, st.C)
        assert_close(y.cpu().numpy(), yo, f"batch {batch} y step {t}")
        kept = np.nonzero(~folded)[0]
        bi, si = torch.from_numpy(kept).cuda(), torch.from_numpy(slot[kept]).cuda()
        np.testing.assert_array_equal(cache.rec_dt[bi, :, si].cpu().numpy(), st.dt[kept])
        np.testing.assert_array_equal(cache.rec_x[bi, :, si].float().cpu().numpy(), st.x[kept])
        np.testing.assert_array_equal(cache.rec_B[bi, :, si].float().cpu().numpy(), st.B[kept])
        np.testing.assert_array_equal(cache.rec_C[bi, :, si].float().cpu().numpy(), st.C[kept])
        for b in np.nonzero(folded)[0]:
            e = rel_err(cache.ckpt[int(b)].cpu().numpy(), orc.h[b])
            assert e <= RTOL, f"folded checkpoint of seq {b} at step {t}: {e:.3e}"
            folded_seqs.add(int(b))
    assert folded_seqs == set(range(batch))        # every sequence took a fused flush
    rs.flush(cache)
    ring.flush()
    _check_ring(cache, ring)
    assert_close(cache.ckpt.cpu().numpy(), orc.h, f"batch {batch} flushed checkpoints")


@pytest.mark.parametrize("chunk", [8, 4])
def test_small_batch_matches_persistent_bit_for_bit(chunk):
    from ssm_decode_state_gb300 import replayssm as rs
    shape, seed = _serving(32)
    prm = gen.mamba2_params(shape, seed)
    h0 = torch.from_numpy(gen.mamba2_random_state(shape, seed)).cuda()
    A, D = torch.from_numpy(prm.A), torch.from_numpy(prm.D)
    dims32 = rs.mamba2_dims(32, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    dimsc = rs.mamba2_dims(chunk, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    whole = rs.mamba2_cache(dims32, A, D, ckpt=h0.clone())
    parts = rs.mamba2_cache(dimsc, A, D, ckpt=h0.clone(), capacity=32)
    lens, heads = _stagger(32, shape.L, shape.L - 1)
    _m2_prefill(whole, shape, prm, seed, lens, heads)
    _m2_prefill(parts, shape, prm, seed, lens, heads)
    maps = [torch.arange(c0, c0 + chunk, dtype=torch.int32).cuda() for c0 in range(0, 32, chunk)]
    for t in range(2 * shape.L + 1):
        dt, x, B, C = _dev(gen.mamba2_step_inputs(shape, prm, seed, t))
        y32 = rs.decode(whole, dt, x, B, C)
        yc = torch.cat([rs.decode(parts, *(v[chunk * i:chunk * i + chunk].contiguous() for v in (dt, x, B, C)),
                                  slots=m)
                        for i, m in enumerate(maps)])
        assert torch.equal(y32, yc), f"y differs at step {t}"
    for f in FIELDS:
        assert torch.equal(getattr(whole, f), getattr(parts, f)), f
    assert int(whole.err.item()) == 0 and int(parts.err.item()) == 0
    assert not parts.arrive.any().item()


@pytest.mark.parametrize("L,lens", [(32, [32, 31, 0]), (1, [1, 0])], ids=["L32_full_ring", "L1"])
def test_small_batch_ring_extremes(L, lens):
    """Ring lengths at the limits: L = 32 with a full ring (len = L, left by a
    verify), so the decode folds L + 1 = 33 records (list position 32 in every
    staging and weight array, a second pass of B . C), and L = 1, where every
    decode folds.  Serving shape, small-batch kernel, against the oracle over a
    few steps, then a standalone flush; ring pointers exact."""
    from ssm_decode_state_gb300 import replayssm as rs
    w = gen.workloads()["mamba2_b256"]
    s = w.shape
    batch = len(lens)
    shape = gen.Mamba2Shape(batch, s.nheads, s.headdim, s.dstate, s.ngroups, L, True)
    seed = w.seed + 1000 + L
    prm = gen.mamba2_params(shape, seed)
    h0 = gen.mamba2_random_state(shape, seed)
    dims = rs.mamba2_dims(batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, L)
    cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D),
                            ckpt=torch.from_numpy(h0).cuda())
    lens = np.array(lens)
    heads = (np.arange(batch) * 7 + 3) % L
    pre = _m2_prefill(cache, shape, prm, seed, lens, heads)
    ring = _ring_model(lens, heads, L)
    orc = Mamba2Stepwise(prm.A, prm.D, shape.ngroups, h0)
    _m2_oracle_prefill(orc, pre, lens, np.arange(batch))
    for t in range(3):
        st = gen.mamba2_step_inputs(shape, prm, seed, t)
        y = rs.decode(cache, *_dev(st))
        folded = np.array([f is not None for f in ring.decode([t] * batch)])
        _check_ring(cache, ring)
        yo = orc.step(st.dt, st.x, st.B, st.C)
        assert_close(y.cpu().numpy(), yo, f"L {L} y step {t}")
        for b in np.nonzero(folded)[0]:
            e = rel_err(cache.ckpt[int(b)].cpu().numpy(), orc.h[b])
            assert e <= RTOL, f"L {L} folded checkpoint of seq {b} at step {t}: {e:.3e}"
    rs.flush(cache)                                # fold what each sequence still buffers
    ring.flush()
    _check_ring(cache, ring)
    assert_close(cache.ckpt.cpu().numpy(), orc.h, f"L {L} flushed checkpoints after 3 steps")
