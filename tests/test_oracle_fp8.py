"""Pins of the FP8 E4M3 encoder and row quantiser."""
import json
import os

import numpy as np
import torch

from oracle.fp8 import dequantize_rows, e4m3_decode, e4m3_encode, quantize_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_e4m3_table.json")


def test_format_table():
    """Code points fixed by the OCP E4M3 definition (tests/golden/fp8_e4m3_table.json)."""
    with open(GOLDEN) as f:
        table = json.load(f)
    for row in table["encode"]:
        v = np.float32(eval(row["value"], {"__builtins__": {}}, {"nan": float("nan"),
                                                                 "inf": float("inf")}))
        assert int(e4m3_encode(np.array([v]))[0]) == int(row["code"], 16), row
    for row in table["decode"]:
        got = float(e4m3_decode(np.array([int(row["code"], 16)], np.uint8))[0])
        want = eval(row["value"], {"__builtins__": {}}, {"nan": float("nan")})
        assert (np.isnan(got) and np.isnan(want)) or got == want, row


def test_all_codes_round_trip():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3_decode(codes)
    finite = ~np.isnan(vals)
    re = e4m3_encode(vals[finite].astype(np.float32))
    # +0 and -0 keep their sign bit; every finite code maps back to itself
    np.testing.assert_array_equal(re, codes[finite])


def test_matches_torch_cast():
    """The library cast rounds to nearest even as well; it does not saturate,
    so compare where the rounded value stays finite (|v| <= 464)."""
    rng = np.random.default_rng(21)
    v = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 10.0,
        rng.standard_normal(100000).astype(np.float32) * 1e-2,
        rng.uniform(-464, 464, 100000).astype(np.float32),
        # exact ties between neighbouring codes in every binade
        (e4m3_decode(np.arange(0, 126, dtype=np.uint8)) / 2
         + e4m3_decode(np.arange(1, 127, dtype=np.uint8)) / 2).astype(np.float32),
    ])
    v = v[np.abs(v) <= 464]
    ours = e4m3_encode(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, lib)


def test_saturation():
    v = np.array([465.0, 1e6, np.inf, -500.0, -np.inf], np.float32)
    np.testing.assert_array_equal(e4m3_encode(v), np.array([0x7E, 0x7E, 0x7E, 0xFE, 0xFE], np.uint8))


def test_row_quantiser_error_bound():
    """Every dequantised value is within half a code step of the float32 value:
    2^-4 relative for normals, 2^-10 * scale below the smallest normal."""
    rng = np.random.default_rng(22)
    h = (rng.standard_normal((64, 128)) * 0.1).astype(np.float32)
    h[3] = 0.0
    h[5, :64] *= 1e-4
    codes, scale = quantize_rows(h)
    assert scale[3] == 1.0 and not codes[3].any()
    back = dequantize_rows(codes, scale).astype(np.float64)
    bound = 2.0 ** -4 * np.abs(h) + 2.0 ** -10 * scale[:, None] + 1e-6 * np.abs(h)
    assert np.all(np.abs(back - h) <= bound)
    # the row maximum maps to the largest code, 448
    amax_idx = np.argmax(np.abs(h), axis=1)
    top = codes[np.arange(64), amax_idx] & 0x7F
    assert np.all(top[np.arange(64) != 3] == 0x7E)
