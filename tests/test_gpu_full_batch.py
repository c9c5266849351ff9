"""Every sequence of the full-size workloads against the oracle.

The other parity tests at serving size let the oracle follow a few sampled
sequences.  Here the oracle follows all of them, so every work item of the
kernels' static schedules (every CTA, every position of an item in a CTA's
list) is checked.  To reach every ring length and a fold within a few steps,
each sequence starts with its own number of buffered records (staggered rings,
the ring head varied too, so runs wrap around the ring end): the records are
drawn from the seeded generator and written into the ring, and the oracle
applies the same tokens stepwise (a sequence that buffers fewer records gets
identity tokens in their place: dt = 0 for Mamba-2, alpha = 1 and beta = 0 for
Gated DeltaNet, which leave the state exactly as it is).

The GPU runs the whole batch and keeps its outputs on the host; the oracle
then runs in chunks of sequences so its float64 state stays small.  A final
standalone flush of every sequence is compared against the oracle's state too.
"""
import numpy as np
import pytest
import torch

from oracle.gdn import GDNStepwise
from oracle.mamba2 import Mamba2Stepwise
from oracle.ring import RingModel
from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL, assert_close, rel_err

pytestmark = pytest.mark.gpu

CHUNK = 64          # sequences per oracle pass


def _stagger(batch, L, lmax):
    """Buffered records per sequence (0..lmax) and ring heads (all of 0..L-1)."""
    b = np.arange(batch)
    return b % (lmax + 1), (5 * b + 3) % L


def _ring_model(lens, heads, L):
    ring = RingModel(len(lens), L)
    for s, n, h in zip(ring.seqs, lens, heads):
        s.head = int(h)
        s.tags = [("pre", j) for j in range(int(n))]
    return ring


def _check_ring(cache, ring):
    np.testing.assert_array_equal(cache.ring_len.cpu().numpy(), ring.lens())
    np.testing.assert_array_equal(cache.ring_head.cpu().numpy(), ring.heads())
    assert int(cache.err.item()) == 0
    assert not cache.arrive.any().item()


# ------------------------------------------------------------------- Mamba-2

def _m2_prefill(cache, shape, prm, seed, lens, heads):
    """Write records j < lens[b] into ring slot (heads[b] + j) mod L; returns the
    per-position inputs for the oracle."""
    pre = []
    for j in range(int(lens.max())):
        st = gen.mamba2_step_inputs(shape, prm, seed, 90_000 + j)
        pre.append(st)
        sel = np.nonzero(lens > j)[0]
        bi = torch.from_numpy(sel).cuda()
        si = torch.from_numpy((heads[sel] + j) % shape.L).cuda()
        cache.rec_dt[bi, :, si] = torch.from_numpy(st.dt[sel]).cuda()
        cache.rec_x[bi, :, si] = torch.from_numpy(st.x[sel]).cuda().to(torch.bfloat16)
        cache.rec_B[bi, :, si] = torch.from_numpy(st.B[sel]).cuda().to(torch.bfloat16)
        cache.rec_C[bi, :, si] = torch.from_numpy(st.C[sel]).cuda().to(torch.bfloat16)
    cache.ring_len.copy_(torch.from_numpy(lens.astype(np.int32)))
    cache.ring_head.copy_(torch.from_numpy(heads.astype(np.int32)))
    return pre


def _m2_oracle_prefill(orc, pre, lens, c):
    for j, st in enumerate(pre):
        dt = st.dt[c].copy()
        dt[lens[c] <= j] = 0.0                      # identity token: exp(0 A) = 1, 0 x B^T = 0
        orc.step(dt, st.x[c], st.B[c], st.C[c])


def _dev(st):
    return (torch.from_numpy(st.dt).cuda(), torch.from_numpy(st.x).cuda().to(torch.bfloat16),
            torch.from_numpy(st.B).cuda().to(torch.bfloat16), torch.from_numpy(st.C).cuda().to(torch.bfloat16))


def test_mamba2_b256_every_sequence():
    """Mamba-2 layer at serving shape, batch 256, rings staggered 0..15 records:
    4 decode steps (every sequence passes 4 ring lengths; a quarter of them take
    the fused flush), y of all 256 sequences and the folded checkpoints against
    the oracle, ring pointers and the appended records exact; then a standalone
    flush of every sequence against the oracle's state."""
    from ssm_decode_state_gb300 import replayssm as rs
    w = gen.workloads()["mamba2_b256"]
    shape, seed = w.shape, w.seed
    prm = gen.mamba2_params(shape, seed)
    h0 = gen.mamba2_random_state(shape, seed)
    dims = rs.mamba2_dims(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D),
                            ckpt=torch.from_numpy(h0).cuda())
    lens, heads = _stagger(shape.batch, shape.L, shape.L - 1)
    pre = _m2_prefill(cache, shape, prm, seed, lens, heads)
    ring = _ring_model(lens, heads, shape.L)
    steps, ys, folds = [], [], []
    for t in range(4):
        st = gen.mamba2_step_inputs(shape, prm, seed, t)
        slot = np.array([(s.head + s.len) % shape.L for s in ring.seqs])
        y = rs.decode(cache, *_dev(st))
        folded = np.array([f is not None for f in ring.decode([t] * shape.batch)])
        _check_ring(cache, ring)
        kept = np.nonzero(~folded)[0]               # the token's record sits in its ring slot
        bi, si = torch.from_numpy(kept).cuda(), torch.from_numpy(slot[kept]).cuda()
        np.testing.assert_array_equal(cache.rec_dt[bi, :, si].cpu().numpy(), st.dt[kept])
        np.testing.assert_array_equal(cache.rec_x[bi, :, si].float().cpu().numpy(), st.x[kept])
        np.testing.assert_array_equal(cache.rec_B[bi, :, si].float().cpu().numpy(), st.B[kept])
        np.testing.assert_array_equal(cache.rec_C[bi, :, si].float().cpu().numpy(), st.C[kept])
        fb = np.nonzero(folded)[0]
        folds.append((fb, cache.ckpt[torch.from_numpy(fb).cuda()].cpu().numpy()))
        steps.append(st)
        ys.append(y.cpu().numpy())
    assert sum(len(f[0]) for f in folds) == shape.batch // 4
    rs.flush(cache)                                 # every sequence: fold what is buffered
    ring.flush()
    _check_ring(cache, ring)
    final = cache.ckpt.cpu().numpy()
    del cache
    worst = {"y": 0.0, "fold": 0.0, "flush": 0.0}
    for c0 in range(0, shape.batch, CHUNK):
        c = np.arange(c0, c0 + CHUNK)
        orc = Mamba2Stepwise(prm.A, prm.D, shape.ngroups, h0[c])
        _m2_oracle_prefill(orc, pre, lens, c)
        for t, st in enumerate(steps):
            yo = orc.step(st.dt[c], st.x[c], st.B[c], st.C[c])
            worst["y"] = max(worst["y"], assert_close(ys[t][c], yo, f"y step {t}, seqs {c0}+"))
            fb, ck = folds[t]
            for i, b in enumerate(fb):
                if c0 <= b < c0 + CHUNK:
                    e = rel_err(ck[i], orc.h[b - c0])
                    assert e <= RTOL, f"folded checkpoint of seq {b} at step {t}: {e:.3e}"
                    worst["fold"] = max(worst["fold"], e)
        for i, b in enumerate(c):
            e = rel_err(final[b], orc.h[i])
            assert e <= RTOL, f"flushed checkpoint of seq {b}: {e:.3e}"
            worst["flush"] = max(worst["flush"], e)
    print("mamba2 b256 every sequence, max errors", worst)


def test_mamba2_verify_b512_every_sequence():
    """Speculative verify at batch 512 (T = 4), rings staggered 0..16 records so
    the sequences holding 13..16 pre-flush: 3 verify + rollback steps, the draft
    outputs of all 512 sequences against the oracle's causal scoring and
    acceptance, ring pointers exact; then a standalone flush of every sequence
    against the oracle's state."""
    from ssm_decode_state_gb300 import replayssm as rs
    w = gen.workloads()["mamba2_verify_b512_T4"]
    shape, seed, T = w.shape, w.seed, w.T
    prm = gen.mamba2_params(shape, seed)
    h0 = gen.mamba2_random_state(shape, seed)
    dims = rs.mamba2_dims(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D),
                            ckpt=torch.from_numpy(h0).cuda())
    lens, heads = _stagger(shape.batch, shape.L, shape.L)
    pre = _m2_prefill(cache, shape, prm, seed, lens, heads)
    ring = _ring_model(lens, heads, shape.L)
    steps, ys, accs = [], [], []
    n_pre = 0
    for t in range(3):
        d = gen.mamba2_draft_inputs(shape, prm, seed, t, T)
        y = rs.verify(cache, *_dev(d))
        n_pre += sum(f is not None for f in ring.verify([[(t, i) for i in range(T)]] * shape.batch))
        acc = gen.accepted_counts(shape.batch, T, seed, t)
        rs.rollback(cache, T, torch.from_numpy(acc).cuda())
        ring.rollback(T, acc)
        _check_ring(cache, ring)
        steps.append(d)
        accs.append(acc)
        ys.append(y.cpu().numpy())
    assert n_pre >= 4 * shape.batch // 17
    rs.flush(cache)
    ring.flush()
    _check_ring(cache, ring)
    final = cache.ckpt.cpu().numpy()
    del cache
    worst = {"y": 0.0, "flush": 0.0}
    for c0 in range(0, shape.batch, CHUNK):
        c = np.arange(c0, c0 + CHUNK)
        orc = Mamba2Stepwise(prm.A, prm.D, shape.ngroups, h0[c])
        _m2_oracle_prefill(orc, pre, lens, c)
        for t, d in enumerate(steps):
            yo, states = orc.verify(d.dt[c], d.x[c], d.B[c], d.C[c])
            worst["y"] = max(worst["y"], assert_close(ys[t][c], yo, f"verify y step {t}, seqs {c0}+"))
            orc.accept(states, accs[t][c])
        for i, b in enumerate(c):
            e = rel_err(final[b], orc.h[i])
            assert e <= RTOL, f"flushed checkpoint of seq {b}: {e:.3e}"
            worst["flush"] = max(worst["flush"], e)
    print("mamba2 verify b512 every sequence, max errors", worst)


# ------------------------------------------------------------ Gated DeltaNet

def _gdn_dev(st):
    return tuple(torch.from_numpy(a).cuda().to(torch.bfloat16) for a in (st.q, st.k, st.v)) + \
        (torch.from_numpy(st.alpha).cuda(), torch.from_numpy(st.beta).cuda())


def test_gdn_b256_every_sequence():
    """Gated DeltaNet layer, batch 256, 32 heads, dk = dv = 128, rings staggered
    0..15 records: 4 decode steps, o of all 256 sequences and the folded
    checkpoints against the oracle, ring pointers exact; then a standalone flush
    of every sequence against the oracle's state."""
    from ssm_decode_state_gb300 import replayssm as rs
    w = gen.workloads()["gdn_b256"]
    shape, seed = w.shape, w.seed
    S0 = gen.gdn_random_state(shape, seed)
    dims = rs.gdn_dims(shape.batch, shape.nheads, shape.dk, shape.dv, shape.L)
    cache = rs.gdn_cache(dims, ckpt=torch.from_numpy(S0).cuda())
    lens, heads = _stagger(shape.batch, shape.L, shape.L - 1)
    pre = []
    for j in range(int(lens.max())):
        st = gen.gdn_step_inputs(shape, seed, 90_000 + j)
        pre.append(st)
        sel = np.nonzero(lens > j)[0]
        bi = torch.from_numpy(sel).cuda()
        si = torch.from_numpy((heads[sel] + j) % shape.L).cuda()
        cache.rec_k[bi, :, si] = torch.from_numpy(st.k[sel]).cuda().to(torch.bfloat16)
        cache.rec_v[bi, :, si] = torch.from_numpy(st.v[sel]).cuda().to(torch.bfloat16)
        cache.rec_alpha[bi, :, si] = torch.from_numpy(st.alpha[sel]).cuda()
        cache.rec_beta[bi, :, si] = torch.from_numpy(st.beta[sel]).cuda()
    cache.ring_len.copy_(torch.from_numpy(lens.astype(np.int32)))
    cache.ring_head.copy_(torch.from_numpy(heads.astype(np.int32)))
    ring = _ring_model(lens, heads, shape.L)
    steps, outs, folds = [], [], []
    for t in range(4):
        st = gen.gdn_step_inputs(shape, seed, t)
        o = rs.gdn_decode(cache, *_gdn_dev(st))
        folded = np.array([f is not None for f in ring.decode([t] * shape.batch)])
        _check_ring(cache, ring)
        fb = np.nonzero(folded)[0]
        folds.append((fb, cache.ckpt[torch.from_numpy(fb).cuda()].cpu().numpy()))
        steps.append(st)
        outs.append(o.cpu().numpy())
    assert sum(len(f[0]) for f in folds) == shape.batch // 4
    rs.gdn_flush(cache)
    ring.flush()
    _check_ring(cache, ring)
    final = cache.ckpt.cpu().numpy()
    del cache
    worst = {"o": 0.0, "fold": 0.0, "flush": 0.0}
    for c0 in range(0, shape.batch, CHUNK):
        c = np.arange(c0, c0 + CHUNK)
        orc = GDNStepwise(S0[c])
        for j, st in enumerate(pre):
            al, be = st.alpha[c].copy(), st.beta[c].copy()
            pad = lens[c] <= j                          # identity token: alpha 1, beta 0
            al[pad], be[pad] = 1.0, 0.0
            orc.step(st.q[c], st.k[c], st.v[c], al, be)
        for t, st in enumerate(steps):
            oo = orc.step(st.q[c], st.k[c], st.v[c], st.alpha[c], st.beta[c])
            worst["o"] = max(worst["o"], assert_close(outs[t][c], oo, f"gdn o step {t}, seqs {c0}+"))
            fb, ck = folds[t]
            for i, b in enumerate(fb):
                if c0 <= b < c0 + CHUNK:
                    e = rel_err(ck[i], orc.S[b - c0])
                    assert e <= RTOL, f"folded checkpoint of seq {b} at step {t}: {e:.3e}"
                    worst["fold"] = max(worst["fold"], e)
        for i, b in enumerate(c):
            e = rel_err(final[b], orc.S[i])
            assert e <= RTOL, f"flushed checkpoint of seq {b}: {e:.3e}"
            worst["flush"] = max(worst["flush"], e)
    print("gdn b256 every sequence, max errors", worst)
