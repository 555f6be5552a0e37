"""Pins for the oracle's MXFP8 decode (E4M3 elements, UE8M0 block scales).

The tables are built from the format's bit fields; these tests tie them to
torch's own float8 types (an independent implementation), to spot values of
the format definition (tests/golden/e4m3_spot_values.txt) and to structural
properties of the format.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import mxfp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_ue8m0_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()


def test_e4m3_table_matches_torch_all_codes():
    ref = torch_e4m3_values()
    ours = oracle.E4M3
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))
    assert set(np.flatnonzero(np.isnan(ours))) == {0x7F, 0xFF}


def test_ue8m0_table_matches_torch_all_codes():
    ref = torch_ue8m0_values()
    ours = oracle.UE8M0
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])


def test_spot_values_from_format_definition():
    path = os.path.join(GOLDEN, "e4m3_spot_values.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kind, code, value = line.split()
        code = int(code, 16)
        table = oracle.E4M3 if kind == "e4m3" else oracle.UE8M0
        got = table[code]
        if value == "nan":
            assert math.isnan(got)
        else:
            want = float.fromhex(value)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (kind, hex(code))
        n += 1
    assert n >= 12


def test_positive_codes_strictly_increase():
    # E4M3 is sign-magnitude with the exponent above the mantissa: codes
    # 0x00..0x7E enumerate the non-negative values in increasing order, and the
    # negative half mirrors them.
    v = oracle.E4M3[:0x7F]
    assert np.all(np.diff(v) > 0)
    assert np.array_equal(oracle.E4M3[0x80:0xFF], -v)
    # consecutive normals within one binade are 1/8 of the binade apart
    for e in range(1, 16):
        base = 2.0 ** (e - 7)
        codes = [(e << 3) | m for m in range(8) if not (e == 15 and m == 7)]
        assert np.allclose(np.diff(oracle.E4M3[codes]), base / 8, rtol=0, atol=0)


def test_all_products_exact():
    # every (code, scale) pair: the oracle's dequantised value equals the
    # product of torch's two decodes (exact in float64: 4 significant bits
    # times a power of two)
    ev = torch_e4m3_values()
    sv = torch_ue8m0_values()
    codes = np.repeat(np.arange(256, dtype=np.uint8), 32)[None, :].repeat(256, 0)  # [256 scales, 256*32]
    scales = np.arange(256, dtype=np.uint8)[:, None].repeat(256, 1)                 # one scale per 32
    got = oracle.dequantize(codes, scales)
    want = ev[codes.astype(np.int64)] * sv[:, None]
    both_nan = np.isnan(got) & np.isnan(want)
    assert np.array_equal(got[~both_nan], want[~both_nan])
    assert np.array_equal(np.isnan(got), np.isnan(want))


def test_block_scale_indexing():
    # K = 128: four blocks, each with its own scale; element K must use block K // 32
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 0x7F, size=(3, 128)).astype(np.uint8)
    scales = rng.integers(100, 150, size=(3, 4)).astype(np.uint8)
    got = oracle.dequantize(codes, scales)
    ev = torch_e4m3_values()
    for r in range(3):
        for K in range(128):
            want = ev[codes[r, K]] * 2.0 ** (int(scales[r, K // 32]) - 127)
            assert got[r, K] == want


def test_subnormal_and_extreme_scales():
    # smallest subnormal code at the smallest scale, largest code at the largest
    assert oracle.dequantize(np.array([[1] * 32], np.uint8), np.array([[0]], np.uint8))[0, 0] == 2.0 ** (-9 - 127)
    assert oracle.dequantize(np.array([[0x7E] * 32], np.uint8), np.array([[254]], np.uint8))[0, 0] == 448.0 * 2.0 ** 127


def test_shape_checks():
    with pytest.raises(ValueError):
        oracle.dequantize(np.zeros((2, 48), np.uint8), np.zeros((2, 1), np.uint8))
    with pytest.raises(ValueError):
        oracle.dequantize(np.zeros((2, 64), np.uint8), np.zeros((2, 3), np.uint8))


def test_closed_form_scalar_decoders_agree_with_tables():
    for c in range(256):
        a, b = mxfp8.e4m3_decode(c), oracle.E4M3[c]
        assert (math.isnan(a) and math.isnan(b)) or a == b
        a, b = mxfp8.ue8m0_decode(c), oracle.UE8M0[c]
        assert (math.isnan(a) and math.isnan(b)) or a == b
