"""Pins of the oracle's FP8 (E4M3) KV-cache rows: the code table and rounding against
torch's float8_e4m3fn, a hand-derived fixture (tests/golden/hand_e4m3_rows.txt), and the
properties the power-of-two row scale fixes."""
import os

import numpy as np
import pytest
import torch

from helpers import from_bits, to_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
f8 = getattr(torch, "float8_e4m3fn", None)


@pytest.mark.skipif(f8 is None, reason="torch without float8_e4m3fn")
def test_e4m3_code_table_matches_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(f8).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2     # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.skipif(f8 is None, reason="torch without float8_e4m3fn")
def test_e4m3_rounding_matches_torch_including_ties(oracle_mod):
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.uniform(-448, 448, 3000), rng.standard_normal(3000),
                        np.exp2(rng.uniform(-12, 8, 3000)) * rng.choice([-1, 1], 3000)])
    # every midpoint between neighbouring finite codes (ties), both signs
    vals = np.array([oracle_mod.e4m3_to_f64(c) for c in range(0x7F)])
    mids = (vals[1:] + vals[:-1]) / 2
    x = np.concatenate([x, mids, -mids]).astype(np.float32)       # all exact in fp32
    ref = torch.from_numpy(x).to(f8).view(torch.uint8).numpy()
    got = np.array([oracle_mod.f64_to_e4m3(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_rows_hand_golden(oracle_mod):
    rows = []
    with open(os.path.join(GOLDEN, "hand_e4m3_rows.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([part.split() for part in line.split(";")])
    for vals, scale, codes, back in rows:
        x = np.array(vals, dtype=np.float64)
        bits = to_bits(x)
        assert np.array_equal(from_bits(bits), x)          # the fixture's inputs are bf16 values
        c, s = oracle_mod.quantize_rows_e4m3(bits[None])
        assert float(s[0]) == float(scale[0])
        assert list(c[0]) == [int(h, 16) for h in codes]
        assert np.array_equal(oracle_mod.dequantize_e4m3(c, s)[0], np.array(back, dtype=np.float64))


def test_e4m3_row_properties(oracle_mod):
    rng = np.random.default_rng(32)
    x = to_bits(rng.standard_normal((200, 128)) * np.exp2(rng.integers(-10, 10, (200, 1))))
    c, s = oracle_mod.quantize_rows_e4m3(x)
    xf = from_bits(x)
    back = oracle_mod.dequantize_e4m3(c, s)
    # scales are powers of two, and the largest element lands in the top binade of E4M3
    # (its value in (224, 448]; its code may round down to 224)
    assert np.all(np.exp2(np.round(np.log2(s))) == s)
    amax = np.abs(xf).max(axis=1)
    top = np.abs(back).max(axis=1) / s
    assert np.all((top >= 224) & (top <= 448)) and np.all(amax <= 448 * s) and np.all(amax > 224 * s)
    # round to nearest: within half a code spacing (relative 2^-4 for normal codes, 2^-10
    # absolute in scaled units for subnormal ones)
    err = np.abs(back - xf) / s[:, None]
    spacing = np.maximum(np.exp2(np.floor(np.log2(np.maximum(np.abs(xf) / s[:, None], 2.0 ** -6))) - 3), 2.0 ** -9)
    assert np.all(err <= spacing / 2 + 1e-300)
    # dequantised values are bf16 values (4 significant bits at most), exactly
    assert np.array_equal(from_bits(to_bits(back)), back)
    # scaling a row by 2^m scales its scale by 2^m and keeps its codes
    x8 = to_bits(xf * 8.0)
    c8, s8 = oracle_mod.quantize_rows_e4m3(x8)
    assert np.array_equal(c8, c) and np.array_equal(s8, s * 8)
