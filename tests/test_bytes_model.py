"""The algorithmic-bytes model against the pages' size arithmetic (Clarity,
Key figures and claim ledger [10], [11], [19]-[21]; AT Pulse, What happened:
replay roughly halves the state traffic)."""
from ssm_decode_state_gb300 import bytes_model as bm


def test_state_size_and_kv_equivalents():
    u = bm.mamba2_units(128, 64, 128, 8)
    assert u.S == 4 * 1024 * 1024                    # 4 MiB FP32 state per sequence and layer
    kv_token = 512                                   # 0.5 KiB FP8 KV entry per token
    assert u.S // kv_token == 8192                   # one SSM layer = 8,192 KV tokens
    assert 5 * u.S // kv_token == 40960              # five SSM layers per attention layer
    assert 2 * 5 * u.S // kv_token == 81920          # load + store every step


def test_replay_roughly_halves_traffic():
    u = bm.mamba2_units(128, 64, 128, 8)
    conv = bm.mamba2_conventional(u)
    assert conv == 8442368
    period = bm.mamba2_replay_period(u, 16)
    assert round(period) == 4671968
    assert 0.5 < period / conv < 0.6
    assert round(bm.mamba2_replay_period(u, 16, read_copy=True)) == 1821152


def test_nvfp4_copy_bytes():
    """NVFP4 copy of one sequence: 4-bit codes (512 KiB), an E4M3 scale per 16
    columns (64 KiB) and a float32 scale per row (32 KiB); every step of a
    period moves the copy once (15 reads, 1 rewrite at the flush), so the
    period mean is the FP8 one less the size difference."""
    u = bm.mamba2_units(128, 64, 128, 8)
    assert u.Sq4 == 524288 + 65536 + 32768 == 622592
    assert round(bm.mamba2_replay_period(u, 16, read_copy=2)) == 1821152 - (1081344 - 622592) == 1362400
    assert bm.mamba2_replay_decode(u, 3, 16, 2) == bm.mamba2_replay_decode(u, 3, 16) - u.S + u.Sq4


def test_fp16_checkpoint_bytes():
    """An FP16 checkpoint (2 MiB per sequence) halves the checkpoint term of
    every step: read on non-flush steps, read and written at the flush."""
    u = bm.mamba2_units(128, 64, 128, 8)
    assert bm.mamba2_replay_decode(u, 3, 16, ckpt_f16=True) == bm.mamba2_replay_decode(u, 3, 16) - 2 * 1024 * 1024
    assert bm.mamba2_replay_decode(u, 15, 16, ckpt_f16=True) == bm.mamba2_replay_decode(u, 15, 16) - 4 * 1024 * 1024
    assert round(bm.mamba2_replay_period(u, 16, ckpt_f16=True)) == 4671968 - (15 * 2 + 4) * 1024 * 1024 // 16
    assert bm.mamba2_conventional_verify(u, 4) == 21186560


def test_gdn_units():
    g = bm.gdn_units(32, 128, 128)
    assert g.S == 2 * 1024 * 1024
    assert bm.gdn_conventional(g) == 4235520
    assert round(bm.gdn_replay_period(g, 16)) == 2409840


def test_gdn_verify_bytes():
    """Verify of T drafts at the batch-256 GDN shape: one 2 MiB checkpoint read,
    a second (the write-back) only on a pre-flush, and T drafts' token bytes."""
    u = bm.gdn_units(32, 128, 128)
    assert u.S == 2 * 1024 * 1024
    base = bm.gdn_verify(u, 0, 4, 16)
    assert base == u.S + 4 * (u.I + u.Y + u.Rw)
    assert bm.gdn_verify(u, 13, 4, 16) - bm.gdn_verify(u, 12, 4, 16) == u.S + u.Rr   # 13 + 4 > 16 pre-flushes


def test_cache_memory_accounting():
    """Per sequence and layer at the serving shape: the 4 MiB checkpoint plus a ring of
    16 records of 20,992 bytes (dt, x, B, C) and 12 bytes of pointers; the read copies
    add their size, an FP16 checkpoint halves the first term.  In 100 GiB of cache for
    24 SSM layers that is 987 replay sequences against 1,066 conventional ones (FP32), and
    1,464 with an FP16 checkpoint and NVFP4 reads."""
    kw = dict(nheads=128, headdim=64, dstate=128, ngroups=8, L=16)
    c = bm.mamba2_cache_bytes(**kw)
    assert c["checkpoint"] == 4 * 1024 * 1024 and c["ring"] == 16 * 20992 and c["pointers"] == 12
    assert c["total"] == 4194304 + 335872 + 12
    assert bm.mamba2_cache_bytes(**kw, read_copy=1)["read_copy"] == 1081344
    assert bm.mamba2_cache_bytes(**kw, read_copy=2, ckpt_f16=True)["total"] == 2097152 + 622592 + 335872 + 12
    fit = bm.sequences_that_fit(100 * 2 ** 30, 24, **kw)
    assert fit == {"replay": 100 * 2 ** 30 // (24 * 4530188), "conventional": 100 * 2 ** 30 // (24 * 4194304)}
    assert fit["replay"] == 987 and fit["conventional"] == 1066
    assert bm.sequences_that_fit(100 * 2 ** 30, 24, **kw, read_copy=2, ckpt_f16=True)["replay"] == \
        100 * 2 ** 30 // (24 * 3055628) == 1464
