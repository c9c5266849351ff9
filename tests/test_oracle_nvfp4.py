"""Pins of the NVFP4 (E2M1 elements, E4M3 block scales, float32 row scale)
encoder and row quantiser (oracle.nvfp4)."""
import json
import os

import numpy as np

import oracle.nvfp4 as nv
from oracle.fp8 import e4m3_decode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_e2m1.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _val(s):
    return float(eval(s, {"__builtins__": {}}, {}))


def test_format_table():
    """The 16 code points and the rounding cases fixed by the E2M1 definition."""
    g = _golden()
    for row in g["decode"]:
        got = float(nv.e2m1_decode(np.array([int(row["code"], 16)], np.uint8))[0])
        want = _val(row["value"])
        assert got == want and np.signbit(got) == np.signbit(want), row
    for row in g["encode"]:
        v = np.array([_val(row["value"])], np.float32)
        assert int(nv.e2m1_encode(v)[0]) == int(row["code"], 16), row


def test_encoder_is_nearest_with_ties_to_even():
    """Brute force: the code of every value on a fine grid (and random values)
    is the nearest of the 8 magnitudes, the even code on a tie, 6 above 6."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rng = np.random.default_rng(5)
    v = np.concatenate([np.arange(-8 * 64, 8 * 64 + 1) / 64.0, rng.uniform(-10, 10, 20000),
                        rng.standard_normal(20000) * 1e-2]).astype(np.float32)
    a = np.abs(v.astype(np.float64))
    dist = np.abs(a[:, None] - mags[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among tied candidates the one with an even code (index == code for magnitudes)
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    idx = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    idx = np.where(a > 6.0, 7, idx)
    want = idx | (np.signbit(v).astype(np.int64) << 3)
    np.testing.assert_array_equal(nv.e2m1_encode(v), want.astype(np.uint8))


def test_all_codes_round_trip():
    codes = np.arange(16, dtype=np.uint8)
    np.testing.assert_array_equal(nv.e2m1_encode(nv.e2m1_decode(codes).astype(np.float32)), codes)


def test_row_worked_example():
    """The hand-worked row of tests/golden/nvfp4_e2m1.json: codes, packed
    bytes, block scales and row scale, exactly."""
    ex = _golden()["row_example"]
    h = np.array([ex["h"]], np.float32)
    codes, sb, s_r = nv.quantize_rows(h)
    np.testing.assert_array_equal(codes[0], [int(c, 16) for c in ex["codes"]])
    np.testing.assert_array_equal(nv.pack_codes(codes)[0], [int(c, 16) for c in ex["packed"]])
    np.testing.assert_array_equal(sb[0], [int(c, 16) for c in ex["block_scales"]])
    assert s_r[0] == np.float32(_val(ex["row_scale"]))
    back = nv.dequantize_rows(codes, sb, s_r)
    np.testing.assert_allclose(back[0], h[0], rtol=1e-6, atol=0)
    stored, s2 = nv.head_copy(h[None])
    np.testing.assert_array_equal(stored[0], [int(c, 16) for c in ex["packed"] + ex["block_scales"]])
    np.testing.assert_array_equal(nv.head_dequantize(stored, s2, 1, 32), back[None])


def test_quantiser_error_bound_and_block_maximum():
    """Every value of a block with a normal E4M3 scale is within one step of
    the block's grid, d_c = e4m3(sb) * s_r (the largest half-gap of the E2M1
    grid is 1, the largest saturation overshoot 0.375: the scale is within 1/16
    of its target); a subnormal block scale may saturate further.  With a
    normal block scale the block maximum takes the largest code, 6; the row
    scale is amax / 2688."""
    rng = np.random.default_rng(23)
    h = (rng.standard_normal((96, 128)) * 0.1).astype(np.float32)
    h[4, 16:32] *= 1e-3                     # a block far below the row maximum
    h[7, :64] *= 1e-5
    codes, sb, s_r = nv.quantize_rows(h)
    back = nv.dequantize_rows(codes, sb, s_r)
    d = np.repeat(e4m3_decode(sb) * s_r[:, None].astype(np.float64), 16, axis=1)
    err = np.abs(back - h)
    # any block: a step of the grid, or the overshoot of a saturated value
    assert np.all(err <= np.maximum(d, np.abs(h) - 6 * d) * (1 + 2.0 ** -20))
    # a block with a normal E4M3 scale never overshoots by more than 0.375 d
    nrm = np.repeat(e4m3_decode(sb) >= 2.0 ** -6, 16, axis=1)
    assert np.all(err[nrm] <= d[nrm] * (1 + 2.0 ** -20))
    # relative: within 1/4 of |h| where |h| / d is in the normal range of E2M1
    big = (np.abs(h) >= d) & nrm
    assert np.all(err[big] <= 0.25 * np.abs(h)[big] * (1 + 2.0 ** -20) + 0.375 * d[big])
    amax = np.max(np.abs(h), axis=1)
    assert np.all(s_r == (amax.astype(np.float64) / 2688.0).astype(np.float32))
    hb = np.abs(h).reshape(96, 8, 16)
    top = np.take_along_axis(codes.reshape(96, 8, 16), hb.argmax(axis=2)[..., None], axis=2)[..., 0] & 0x7
    normal = e4m3_decode(sb) >= 2.0 ** -6
    assert np.all(top[normal] == 7)
    # the row maximum's block scale is 448 (0x7E), the largest E4M3 value
    blk = np.abs(h).argmax(axis=1) // 16
    assert np.all(sb[np.arange(96), blk] == 0x7E)


def test_zero_and_tiny_rows():
    """A zero row stores zero codes, zero block scales and row scale 0; a row
    below the float32 range of the scales is stored as zero as well."""
    h = np.zeros((3, 32), np.float32)
    h[1] = -0.0
    h[2, 3] = 1e-44                        # 2688 * s_r underflows: s_r = 0
    codes, sb, s_r = nv.quantize_rows(h)
    assert not sb.any() and not s_r.any()
    assert np.all(nv.dequantize_rows(codes, sb, s_r) == 0)
    assert np.all((codes & 0x7) == 0)
