"""FP8 read copy, Gated DeltaNet, device-side error reporting, and the
persistent decode kernel's shape variants."""
import numpy as np
import pytest
import torch

from oracle.fp8 import quantize_rows
from oracle.gdn import GDNStepwise
from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import RTOL, RTOL_INPLACE, assert_close, rel_err, to_dev

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------------- FP8

def test_requant_matches_oracle_bitwise():
    """The read copy built from an FP32 checkpoint equals the oracle's E4M3
    quantisation of the same values, codes and scales bit for bit (including
    a zero row, a row of tiny values and saturating values)."""
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.Mamba2Shape(batch=3, nheads=4, headdim=64, dstate=128, ngroups=1, L=16)
    h0 = gen.mamba2_random_state(shape, 91)
    h0[0, 0, 3] = 0.0
    h0[1, 2, 5] *= 1e-30
    h0[2, 1, 7, :5] = 1e6
    prm = gen.mamba2_params(shape, 91)
    dims = rs.mamba2_dims(3, 4, 64, 128, 1, 16, read_copy=1)
    c = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D), ckpt=to_dev(h0))
    rs.requant(c)
    codes, scale = quantize_rows(h0)
    np.testing.assert_array_equal(c.ckpt_q.cpu().numpy(), codes)
    np.testing.assert_array_equal(c.ckpt_scale.cpu().numpy(), scale)


def _fp8_bound(h32, scale, C, decay):
    """Per row: decay * sum_n |C_n| (2^-4 |h_n| + 2^-10 s), the E4M3 rounding
    bound (half a code step: 2^-4 relative for normals, 2^-10 * scale below
    the smallest normal).  h32 [b,H,P,N], scale [b,H,P], C [b,H,N], decay [b,H]."""
    e = np.abs(h32.astype(np.float64)) * 2.0 ** -4 + 2.0 ** -10 * scale[..., None].astype(np.float64)
    return decay[..., None] * np.einsum("bhpn,bhn->bhp", e, np.abs(C))


def test_fp8_read_copy_b256():
    """Serving shape at batch 256, 1024 decode steps with the FP8 read copy:
    per-step error of y against the FP32 oracle stays within the E4M3 bound;
    the FP32 checkpoint of the FP8 run equals that of an FP32-read run bit for
    bit at every flush (reads never feed the recurrence); the error does not
    drift across the 64 flush windows."""
    from ssm_decode_state_gb300 import replayssm as rs
    from tests.m2_runner import M2Run
    w = gen.workloads()["mamba2_fp8read_b256"]
    sample = [7, 200]
    h0 = gen.mamba2_random_state(w.shape, w.seed)
    r8 = M2Run(w.shape, w.seed, h0=h0, read_copy=1, sample=sample, conventional=False)
    r32 = M2Run(w.shape, w.seed, h0=h0, read_copy=0, sample=[0], conventional=False,
                h0_sample=h0[:1])
    del h0
    prm = r8.params
    g = np.arange(w.shape.nheads) // (w.shape.nheads // w.shape.ngroups)
    errs = []
    for t in range(w.steps):
        st = gen.mamba2_step_inputs(w.shape, prm, w.seed, t)
        dt, x, B, C = r8.dev_inputs(st)
        # checkpoint and read copy as the kernel sees them before this step
        ln = int(r8.cache.ring_len[0].item())
        ck = r8.cache.ckpt[sample].cpu().numpy()
        q = r8.cache.ckpt_q[sample].cpu().numpy()
        sc = r8.cache.ckpt_scale[sample].cpu().numpy()
        y8 = rs.decode(r8.cache, dt, x, B, C)
        rs.decode(r32.cache, dt, x, B, C)
        yo = r8.oracle.step(*r8._slice(st))
        r8.ring.decode([t] * w.shape.batch)
        y8s = y8.cpu().numpy()[sample]
        if ln + 1 < w.shape.L:
            # decay exp(A * sum of dt since the checkpoint), from the inputs
            S = np.zeros((len(sample), w.shape.nheads))
            dts = [r8.tokens[k].dt[sample] for k in sorted(r8.tokens)][-ln:] if ln else []
            for d_ in dts + [st.dt[sample]]:
                S += d_
            decay = np.exp(prm.A[None].astype(np.float64) * S)
            bound = _fp8_bound(ck, sc, st.C[sample][:, g], decay)
            tau = 1e-2 * np.sqrt(np.mean(yo ** 2))
            slack = 1e-4 * np.maximum(np.abs(yo), tau)
            assert np.all(np.abs(y8s - yo) <= bound + slack), f"fp8 bound violated at step {t}"
            assert np.all((q & 0x7F) != 0x7F)                  # no NaN codes
        else:
            # flush step: y from the FP32 values, FP32 checkpoints identical
            np.testing.assert_array_equal(r8.cache.ckpt[sample].cpu().numpy(),
                                          r32.cache.ckpt[sample].cpu().numpy())
        r8._keep(t, st)
        errs.append(np.linalg.norm(y8s - yo) / np.linalg.norm(yo))
    errs = np.array(errs)
    win = errs.reshape(-1, w.shape.L).mean(axis=1)
    assert win[-8:].mean() <= 1.5 * win[:8].mean(), (win[:8].mean(), win[-8:].mean())
    assert errs.max() < 0.1
    print("fp8 per-step normwise rel err of y: mean %.3e max %.3e; per flush window: first 8 %.3e, "
          "last 8 %.3e, max %.3e" % (errs.mean(), errs.max(), win[:8].mean(), win[-8:].mean(), win.max()))


# ----------------------------------------------------------------------- GDN

class GDNRun:
    def __init__(self, shape, seed, sample=None):
        from ssm_decode_state_gb300 import replayssm as rs
        self.rs, self.shape, self.seed = rs, shape, seed
        b = shape.batch
        self.sample = np.arange(b) if sample is None else np.asarray(sample)
        S0 = gen.gdn_random_state(shape, seed)
        self.dims = rs.gdn_dims(b, shape.nheads, shape.dk, shape.dv, shape.L)
        self.cache = rs.gdn_cache(self.dims, ckpt=to_dev(S0))
        self.conv = to_dev(S0)
        self.oracle = GDNStepwise(S0[self.sample])
        self.len = 0
        self.max_err = 0.0

    def step(self, t):
        st = gen.gdn_step_inputs(self.shape, self.seed, t)
        q, k, v = (to_dev(a, torch.bfloat16) for a in (st.q, st.k, st.v))
        al, be = to_dev(st.alpha), to_dev(st.beta)
        o = self.rs.gdn_decode(self.cache, q, k, v, al, be)
        oc = self.rs.gdn_conventional_decode(self.dims, self.conv, q, k, v, al, be)
        s = self.sample
        oo = self.oracle.step(st.q[s], st.k[s], st.v[s], st.alpha[s], st.beta[s])
        # the replay path (output, fold) takes the FP32 gate; the in-place
        # comparison path rounds its state every token and takes its own
        e = assert_close(o.cpu().numpy()[s], oo, f"gdn replay o step {t}", RTOL)
        self.max_err = max(self.max_err, e)
        assert_close(oc.cpu().numpy()[s], oo, f"gdn conventional o step {t}", RTOL_INPLACE)
        fold = self.len + 1 >= self.shape.L
        self.len = 0 if fold else self.len + 1
        assert (self.cache.ring_len.cpu().numpy() == self.len).all()
        assert int(self.cache.err.item()) == 0
        if fold:
            e = rel_err(self.cache.ckpt.cpu().numpy()[s], self.oracle.S)
            assert e <= RTOL, f"gdn checkpoint after step {t}: {e:.3e}"


@pytest.mark.parametrize("dk,dv,L", [(16, 16, 4), (32, 24, 16), (64, 64, 8)])
def test_gdn_small(dk, dv, L):
    shape = gen.GDNShape(batch=3, nheads=4, dk=dk, dv=dv, L=L)
    r = GDNRun(shape, 300 + dk)
    for t in range(3 * L + 1):
        r.step(t)


def test_gdn_flush_standalone():
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.GDNShape(batch=3, nheads=4, dk=32, dv=32, L=8)
    r = GDNRun(shape, 404)
    for t in range(5):
        r.step(t)
    rs.gdn_flush(r.cache, torch.tensor([1, 0, 1], dtype=torch.uint8, device="cuda"))
    assert r.cache.ring_len.cpu().tolist() == [0, 5, 0]
    assert r.cache.ring_head.cpu().tolist() == [5, 0, 5]
    ck = r.cache.ckpt.cpu().numpy()
    for b in (0, 2):
        assert rel_err(ck[b], r.oracle.S[b]) <= RTOL


def test_gdn_b256_sampled():
    """Gated DeltaNet layer, batch 256, 32 heads, dk = dv = 128, L = 16, 256
    steps; the oracle follows 2 sequences."""
    w = gen.workloads()["gdn_b256"]
    r = GDNRun(w.shape, w.seed, sample=[3, 250])
    for t in range(w.steps):
        r.step(t)
    print("gdn b256 max replay error", r.max_err)


# ------------------------------------------------------------ device errors

def test_bad_ring_pointers_skip_sequence():
    from ssm_decode_state_gb300 import replayssm as rs
    from tests.m2_runner import M2Run
    for b_, H, P in [(3, 8, 32), (64, 128, 64), (4, 128, 64)]:   # per-tile, persistent, small-batch kernels
        shape = gen.Mamba2Shape(batch=b_, nheads=H, headdim=P, dstate=128 if P == 64 else 64,
                                ngroups=2, L=8)
        h0 = gen.mamba2_random_state(shape, 5)
        r = M2Run(shape, 5, h0=h0, sample=[0], conventional=False)
        r.decode(0)
        r.cache.ring_len[1] = 9                            # > L
        before = r.cache.ckpt[1].clone()
        rx = r.cache.rec_x[1].clone()
        st = gen.mamba2_step_inputs(shape, r.params, 5, 1)
        rs.decode(r.cache, *r.dev_inputs(st))
        torch.cuda.synchronize()
        assert int(r.cache.err.item()) & rs.DEVERR_RING_META
        assert r.cache.ring_len[1].item() == 9
        assert torch.equal(r.cache.ckpt[1], before) and torch.equal(r.cache.rec_x[1], rx)
        assert r.cache.ring_len[0].item() == 2 and not r.cache.arrive.any().item()


def test_bounded_wait_gives_up_and_reports():
    """Every wait in the persistent kernels is bounded.  Through the test hook,
    the consumer warps' first wait runs out (a barrier nothing arrives on): the
    call returns after about 2 s with the timeout bit set, every copy the
    kernel started has landed, the context stays usable, and a decode on a
    fresh cache afterwards is exact against the oracle."""
    import time
    from ssm_decode_state_gb300 import replayssm as rs
    from tests.m2_runner import M2Run
    shape = gen.Mamba2Shape(batch=8, nheads=128, headdim=64, dstate=128, ngroups=8, L=16)
    h0 = gen.mamba2_random_state(shape, 12)
    r = M2Run(shape, 12, h0=h0, sample=[0], conventional=False)
    st = gen.mamba2_step_inputs(shape, r.params, 12, 0)
    torch.cuda.synchronize()
    t0 = time.time()
    rs.stalled_decode(r.cache, *r.dev_inputs(st))
    torch.cuda.synchronize()
    took = time.time() - t0
    assert int(r.cache.err.item()) & rs.DEVERR_TIMEOUT
    assert 1.0 < took < 60.0, took
    del r
    fresh = M2Run(shape, 12, h0=h0, sample=[0, 7], conventional=False)
    for t in range(3):
        fresh.decode(t)                    # y against the oracle; err word and counters clean


def test_rollback_out_of_range():
    from ssm_decode_state_gb300 import replayssm as rs
    shape = gen.Mamba2Shape(batch=3, nheads=4, headdim=16, dstate=16, ngroups=1, L=8)
    prm = gen.mamba2_params(shape, 1)
    dims = rs.mamba2_dims(3, 4, 16, 16, 1, 8)
    c = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D))
    d = gen.mamba2_draft_inputs(shape, prm, 1, 0, 3)
    rs.verify(c, to_dev(d.dt), to_dev(d.x, torch.bfloat16), to_dev(d.B, torch.bfloat16),
              to_dev(d.C, torch.bfloat16))
    rs.rollback(c, 3, torch.tensor([4, 1, -1], dtype=torch.int32, device="cuda"))
    assert c.ring_len.cpu().tolist() == [3, 1, 3]
    assert int(c.err.item()) == rs.DEVERR_ROLLBACK


# ------------------------------------------- persistent decode shape variants

@pytest.mark.parametrize("batch,L", [(1, 16), (2, 4), (5, 16), (64, 4), (40, 32), (128, 16), (16, 1)])
def test_persistent_variants(batch, L):
    """Serving head shape at batches that pick 1 (batch 1), 2 (batch 2), 4 (batch 5)
    and 8 heads per work item (fewer work items than SMs at batches 1-5), ring lengths
    4..32 (32 lowers the pipeline depth), and L = 1: every step folds its only
    record, which makes replay the conventional recurrence."""
    from tests.m2_runner import M2Run
    shape = gen.Mamba2Shape(batch=batch, nheads=128, headdim=64, dstate=128, ngroups=8, L=L)
    h0 = gen.mamba2_random_state(shape, 21)
    r = M2Run(shape, 21, h0=h0, sample=[0, batch - 1], conventional=False)
    for t in range(2 * L + 3):
        r.decode(t)
        if t % 5 == 0:
            r.check_records(seqs=[0, batch - 1])


def test_persistent_fp8_small_batch():
    """FP8 read copy through the persistent kernel with frequent flushes: ring
    pointers stay exact and, after the flushes, the read copy encodes the new
    FP32 checkpoint to within half an E4M3 step per element."""
    from tests.m2_runner import M2Run
    shape = gen.Mamba2Shape(batch=16, nheads=128, headdim=64, dstate=128, ngroups=8, L=4)
    h0 = gen.mamba2_random_state(shape, 8)
    r = M2Run(shape, 8, h0=h0, read_copy=1, sample=[3], conventional=False)
    for t in range(9):
        r.decode(t, check=False)
        r.check_ring()
    ck = r.cache.ckpt.cpu().numpy().astype(np.float64)
    sc = r.cache.ckpt_scale.cpu().numpy().astype(np.float64)
    codes = r.cache.ckpt_q.cpu().numpy()
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e, m = (codes >> 3) & 0xF, codes & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7))
    dq = sign * mag * sc[..., None]
    bound = 2.0 ** -4 * np.abs(ck) + 2.0 ** -10 * sc[..., None] + 1e-6 * np.abs(ck)
    assert np.all(np.abs(dq - ck) <= bound)


@pytest.mark.parametrize("batch", [64, 128])
def test_persistent_fp8_decodes_every_code_exactly(batch):
    """The FP8 read path decodes every finite E4M3 code exactly.  The copy is
    written directly: row (b, h, p) column n holds code (row index + 3n) mod 256
    (the two NaN codes replaced by 0), row scales are powers of two, C_t is
    one-hot on a column per (b, g), x_t = 0 and dt = 0, so y must equal the
    code's value times the row scale bit for bit (batch 64 takes 4 heads per
    work item, one stage per item; 128 takes 8 heads, two stages per item)."""
    from oracle.fp8 import e4m3_decode
    from ssm_decode_state_gb300 import replayssm as rs
    Bt, H, P, N, G, L = batch, 128, 64, 128, 8, 16
    dims = rs.mamba2_dims(Bt, H, P, N, G, L, read_copy=1)
    cache = rs.mamba2_cache(dims, torch.full((H,), -0.5), torch.zeros(H))
    rows = np.arange(Bt * H * P, dtype=np.int64).reshape(Bt, H, P, 1)
    codes = ((rows + 3 * np.arange(N).reshape(1, 1, 1, N)) % 256).astype(np.uint8)
    codes[(codes == 0x7F) | (codes == 0xFF)] = 0
    scale = (2.0 ** ((np.arange(P) % 7) - 3)).astype(np.float32)
    scale = np.broadcast_to(scale, (Bt, H, P)).copy()
    cache.ckpt_q.copy_(torch.from_numpy(codes))
    cache.ckpt_scale.copy_(torch.from_numpy(scale))
    n0 = (np.arange(Bt).reshape(Bt, 1) * 5 + np.arange(G).reshape(1, G) * 11) % N      # [b, g]
    C = np.zeros((Bt, G, N), np.float32)
    C[np.arange(Bt)[:, None], np.arange(G)[None, :], n0] = 1.0
    rng = np.random.default_rng(5)
    Bm = rng.standard_normal((Bt, G, N)).astype(np.float32)
    dt = torch.zeros(Bt, H, device="cuda")
    x = torch.zeros(Bt, H, P, dtype=torch.bfloat16, device="cuda")
    y = rs.decode(cache, dt, x, to_dev(Bm, torch.bfloat16), to_dev(C, torch.bfloat16))
    torch.cuda.synchronize()
    assert int(cache.err.item()) == 0
    g_of_h = np.arange(H) // (H // G)
    col = n0[:, g_of_h]                                                      # [b, h]
    picked = np.take_along_axis(codes, col[:, :, None, None].repeat(P, axis=2), axis=3)[..., 0]
    expect = e4m3_decode(picked) * scale
    assert len(np.unique(picked)) == 254
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.float64), expect)


# ------------------------------------------- persistent gated-delta decode

class GDNPersistRun:
    """Serving head shape (dk = dv = 128): replay decode, optional standalone
    flushes, against the stepwise oracle on sampled sequences, with a per-
    sequence ring model (head, len) and checks of the appended records."""

    def __init__(self, batch, L, seed, sample):
        from ssm_decode_state_gb300 import replayssm as rs
        self.rs = rs
        self.shape = gen.GDNShape(batch=batch, nheads=32, dk=128, dv=128, L=L)
        self.seed, self.sample = seed, np.asarray(sample)
        S0 = gen.gdn_random_state(self.shape, seed)
        self.dims = rs.gdn_dims(batch, 32, 128, 128, L)
        self.cache = rs.gdn_cache(self.dims, ckpt=to_dev(S0))
        self.oracle = GDNStepwise(S0[self.sample])
        self.head = np.zeros(batch, np.int64)
        self.len = np.zeros(batch, np.int64)

    def step(self, t):
        L = self.shape.L
        st = gen.gdn_step_inputs(self.shape, self.seed, t)
        o = self.rs.gdn_decode(self.cache, *(to_dev(a, torch.bfloat16) for a in (st.q, st.k, st.v)),
                               to_dev(st.alpha), to_dev(st.beta))
        s = self.sample
        oo = self.oracle.step(st.q[s], st.k[s], st.v[s], st.alpha[s], st.beta[s])
        assert_close(o.cpu().numpy()[s], oo, f"gdn persistent o step {t}", RTOL)
        fold = self.len + 1 >= L
        slot = (self.head + self.len) % L
        self.head = np.where(fold, (self.head + self.len + 1) % L, self.head)
        self.len = np.where(fold, 0, self.len + 1)
        np.testing.assert_array_equal(self.cache.ring_len.cpu().numpy(), self.len)
        np.testing.assert_array_equal(self.cache.ring_head.cpu().numpy(), self.head)
        assert int(self.cache.err.item()) == 0
        # the token's records sit in the ring slot it was appended to (non-fold sequences)
        bs = [b for b in s if not fold[b]]
        if bs:
            rk = self.cache.rec_k.cpu().float().numpy()
            rv = self.cache.rec_v.cpu().float().numpy()
            ra = self.cache.rec_alpha.cpu().numpy()
            for b in bs:
                np.testing.assert_array_equal(rk[b, :, slot[b]], bf16_round(st.k[b]))
                np.testing.assert_array_equal(rv[b, :, slot[b]], bf16_round(st.v[b]))
                np.testing.assert_array_equal(ra[b, :, slot[b]], st.alpha[b])
        for i, b in enumerate(s):
            if fold[b]:
                e = rel_err(self.cache.ckpt[b].cpu().numpy(), self.oracle.S[i])
                assert e <= RTOL, f"gdn checkpoint of seq {b} after step {t}: {e:.3e}"

    def flush(self, mask):
        self.rs.gdn_flush(self.cache, torch.tensor(mask, dtype=torch.uint8, device="cuda"))
        m = np.asarray(mask, bool) & (self.len > 0)
        self.head = np.where(m, (self.head + self.len) % self.shape.L, self.head)
        self.len = np.where(m, 0, self.len)
        np.testing.assert_array_equal(self.cache.ring_len.cpu().numpy(), self.len)
        np.testing.assert_array_equal(self.cache.ring_head.cpu().numpy(), self.head)


def bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("batch,L", [(16, 4), (16, 16), (40, 8)])
def test_gdn_persistent_variants(batch, L):
    """Persistent gated-delta decode (serving head shape) at batches of 512 and
    1280 heads, rings of 4..16: outputs and folded checkpoints against the
    oracle, ring pointers and appended records exact."""
    r = GDNPersistRun(batch, L, 610 + L, sample=[0, batch // 2, batch - 1])
    for t in range(2 * L + 3):
        r.step(t)


def test_gdn_persistent_with_standalone_flush():
    """Persistent decodes around a masked standalone flush: the flushed and the
    unflushed sequences then fold at different steps of the same launches."""
    r = GDNPersistRun(16, 8, 77, sample=[0, 1, 5])
    for t in range(3):
        r.step(t)
    r.flush([1, 0] * 8)
    for i, b in enumerate(r.sample):
        if b % 2 == 0:
            assert rel_err(r.cache.ckpt[b].cpu().numpy(), r.oracle.S[i]) <= RTOL
    for t in range(3, 14):
        r.step(t)


def test_gdn_persistent_bad_ring_pointers():
    """A sequence with invalid ring pointers is flagged and left untouched by
    the persistent kernel; the others proceed."""
    r = GDNPersistRun(16, 8, 91, sample=[0])
    r.step(0)
    r.cache.ring_len[3] = 9                               # > L
    before = r.cache.ckpt[3].clone()
    rk = r.cache.rec_k[3].clone()
    st = gen.gdn_step_inputs(r.shape, r.seed, 1)
    r.rs.gdn_decode(r.cache, *(to_dev(a, torch.bfloat16) for a in (st.q, st.k, st.v)),
                    to_dev(st.alpha), to_dev(st.beta))
    torch.cuda.synchronize()
    assert int(r.cache.err.item()) & r.rs.DEVERR_RING_META
    assert r.cache.ring_len[3].item() == 9
    assert torch.equal(r.cache.ckpt[3], before) and torch.equal(r.cache.rec_k[3], rk)
    assert r.cache.ring_len[0].item() == 2 and not r.cache.arrive.any().item()


def test_gdn_cuda_core_fold_when_items_exceed_fold_plan():
    """More than 512 (sequence, head) items per CTA (batch 2 with enough heads
    for this GPU's SM count): the tensor-core fold phase's plan leaves no room
    for the per-item lists, so the decode phase folds on the CUDA cores.  Ring
    of 4, five decodes through a fused flush: outputs and folded checkpoints of
    sampled heads against the oracle, ring pointers exact."""
    from ssm_decode_state_gb300 import replayssm as rs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = (513 * sms + 1) // 2 + 1                      # ceil(2 H / sms) > 512
    L, seed = 4, 919
    shape = gen.GDNShape(batch=2, nheads=H, dk=128, dv=128, L=L)
    g = torch.Generator(device="cuda").manual_seed(seed)
    S0 = torch.randn(2, H, 128, 128, device="cuda", generator=g).mul_(0.1)
    heads = np.array([0, 1, H // 2, H - 1])
    oracle = GDNStepwise(S0[:, torch.from_numpy(heads).cuda()].cpu().numpy())
    cache = rs.gdn_cache(rs.gdn_dims(2, H, 128, 128, L), ckpt=S0)
    for t in range(L + 1):
        st = gen.gdn_step_inputs(shape, seed, t)
        o = rs.gdn_decode(cache, *(to_dev(a, torch.bfloat16) for a in (st.q, st.k, st.v)),
                          to_dev(st.alpha), to_dev(st.beta))
        sel = lambda a: a[:, heads]                   # noqa: E731
        oo = oracle.step(sel(st.q), sel(st.k), sel(st.v), sel(st.alpha), sel(st.beta))
        assert_close(o[:, torch.from_numpy(heads).cuda()].cpu().numpy(), oo, f"o step {t}", RTOL)
        ln = (t + 1) % L
        np.testing.assert_array_equal(cache.ring_len.cpu().numpy(), [ln, ln])
        np.testing.assert_array_equal(cache.ring_head.cpu().numpy(), [0, 0])   # a full fold wraps to 0
        assert int(cache.err.item()) == 0
        if t == L - 1:                                # the fused flush
            ck = cache.ckpt[:, torch.from_numpy(heads).cuda()].cpu().numpy()
            e = rel_err(ck, oracle.S)
            assert e <= RTOL, f"folded checkpoints: {e:.3e}"
