"""Pins for the oracle's MXFP4 decode (E2M1 elements two to a byte, UE8M0
block scales) and for the MXFP4 form of its layer.

The E2M1 table is built from the format's bit fields. These tests tie it to
the format definition's spot values (tests/golden/e2m1_spot_values.txt), to
torch's float8_e4m3fn decode through the exact embedding of E2M1 in E4M3
(sign kept, exponent field + 6, mantissa bit moved to the top of the three),
the nibble unpacking to a scalar loop, and the MXFP4 layer to the MXFP8 layer
on the embedded codes (every E2M1 value is an E4M3 value, the scales are
shared, so the two layers are the same function of the same numbers).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import mxfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def e2m1_to_e4m3_code(c: int) -> int:
    """The E4M3 bit pattern with the same value as E2M1 code c."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    if e == 0 and m == 0:
        return s << 7                      # +-0
    if e == 0:
        return (s << 7) | (6 << 3)         # 0.5 = 2^-1: E4M3 exponent field 6, mantissa 0
    return (s << 7) | ((e + 6) << 3) | (m << 2)


EMBED = np.array([e2m1_to_e4m3_code(c) for c in range(16)], dtype=np.uint8)


def test_e2m1_spot_values_from_format_definition():
    seen = set()
    for line in open(os.path.join(GOLDEN, "e2m1_spot_values.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, value = line.split()
        code = int(code, 16)
        want = float.fromhex(value)
        got = oracle.E2M1[code]
        assert got == want and np.signbit(got) == np.signbit(want), (code, got, want)
        seen.add(code)
    assert seen == set(range(16))


def test_e2m1_matches_torch_e4m3_through_embedding():
    ref = torch.from_numpy(EMBED.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.E2M1, ref)
    assert np.array_equal(np.signbit(oracle.E2M1), np.signbit(ref))


def test_e2m1_structure():
    t = oracle.E2M1
    assert np.all(np.isfinite(t))
    assert np.array_equal(t[8:], -t[:8])
    assert np.all(np.diff(t[:8]) > 0)                 # codes 0..7 increase
    assert t[7] == 6.0 and t[1] == 0.5


def test_unpack_and_dequantize_scalar_loop():
    rng = np.random.default_rng(7)
    R, K = 3, 96
    packed = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    scales = rng.integers(100, 150, size=(R, K // 32), dtype=np.uint8)
    got = mxfp4.dequantize(packed, scales)
    for r in range(R):
        for i in range(K):
            byte = int(packed[r, i // 2])
            code = (byte >> 4) if i % 2 else (byte & 0xF)
            want = oracle.e2m1_decode(code) * 2.0 ** (int(scales[r, i // 32]) - 127)
            assert got[r, i] == want, (r, i)


def test_dequantize_rejects_bad_shapes():
    with pytest.raises(ValueError):
        mxfp4.dequantize(np.zeros((2, 16), np.uint8), np.zeros((2, 2), np.uint8))
    with pytest.raises(ValueError):
        mxfp4.dequantize(np.zeros((2, 8), np.uint8), np.zeros((2, 1), np.uint8))


def _as_mxfp8(expert):
    """An MXFP4 expert's tensors with every code re-expressed as E4M3 bytes."""
    wgu, sgu, wd, sd = expert
    return EMBED[mxfp4.unpack(wgu)], sgu, EMBED[mxfp4.unpack(wd)], sd


def test_mxfp4_layer_equals_mxfp8_layer_on_embedded_codes():
    w = W.workload(0)
    seed = W.seed_of(0)
    T = 3
    x = W.bf16_bits_to_f64(W.make_x(w, seed, T=T))
    ids, wt = oracle.route(W.make_logits(w, seed, T=T).astype(np.float64), w.k)
    ids[1, 1] = w.E + 3           # an out-of-range id contributes nothing in both
    experts = W.make_experts(w, seed, range(w.E), fmt="mxfp4")
    ex8 = {e: _as_mxfp8(t) for e, t in experts.items()}
    a = oracle.layer(x, ids, wt, experts, w.E, w.H, w.I, fmt="mxfp4")
    b = oracle.layer(x, ids, wt, ex8, w.E, w.H, w.I, fmt="mxfp8")
    for key in ("h_spec", "h_pure", "y_spec", "y_pure"):
        assert np.array_equal(a[key], b[key]), key
    assert np.any(a["y_spec"] != 0)


def test_unknown_format_rejected():
    with pytest.raises(ValueError):
        oracle.gate_up(np.zeros((1, 32)), np.zeros((1, 1), np.int64), {}, 1, 32, fmt="fp6")


# ---- the seeded MXFP4 encoder (workloads), checked against brute force ----

def test_encode_mxfp4_picks_nearest_value():
    rng = np.random.default_rng(3)
    a = (rng.standard_normal((4, 64)) * 0.02).astype(np.float32)
    a[0, :32] = 0.0                                    # an all-zero block
    a[1, 5] = 1e-30                                    # a tiny element beside normal ones
    packed, scales = W.encode_mxfp4(a)
    got = mxfp4.dequantize(packed, scales)
    grid = np.unique(np.abs(oracle.E2M1))
    for r in range(a.shape[0]):
        for b in range(2):
            blk = a[r, 32 * b:32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            s = int(scales[r, b]) - 127
            if amax == 0:
                assert s == 0
                assert np.all(got[r, 32 * b:32 * b + 32] == 0)
                continue
            assert 4.0 <= amax / 2.0 ** s < 8.0          # floor(log2 amax) - 2
            for i in range(32):
                q = min(abs(blk[i]) / 2.0 ** s, 6.0)
                d = np.abs(grid - q)
                best = grid[d == d.min()]
                v = abs(got[r, 32 * b + i]) / 2.0 ** s
                assert v in best, (r, b, i, q, v)
                if len(best) == 2:                       # a tie goes to the even code
                    assert v == best[int(np.flatnonzero(grid == best[0])[0] % 2 != 0)]
                if got[r, 32 * b + i] != 0:
                    assert np.sign(got[r, 32 * b + i]) == np.sign(blk[i])


def test_make_expert_mxfp4_shapes_and_bytes():
    w = W.workload(0)
    wgu, sgu, wd, sd = W.make_expert(w, W.seed_of(0), 2, fmt="mxfp4")
    assert wgu.shape == (2 * w.I, w.H // 2) and sgu.shape == (2 * w.I, w.H // 32)
    assert wd.shape == (w.H, w.I // 2) and sd.shape == (w.H, w.I // 32)
    assert w.weight_bytes("mxfp4") == wgu.size + sgu.size + wd.size + sd.size
    assert w.weight_bytes("mxfp8") == w.weight_bytes_per_expert


def _scalar_loop_agrees(dq):
    rng = np.random.default_rng(11)
    packed = rng.integers(0, 256, size=(2, 64), dtype=np.uint8)
    scales = rng.integers(110, 140, size=(2, 4), dtype=np.uint8)
    got = dq(packed, scales)
    for r in range(2):
        for i in range(128):
            byte = int(packed[r, i // 2])
            code = (byte >> 4) if i % 2 else (byte & 0xF)
            if got[r, i] != oracle.e2m1_decode(code) * 2.0 ** (int(scales[r, i // 32]) - 127):
                return False
    return True


def test_pins_catch_planted_mxfp4_mistakes():
    # a swapped nibble order and a scale indexed per packed byte, planted in
    # copies of the oracle's decode, must each fail the scalar-loop pin
    assert _scalar_loop_agrees(mxfp4.dequantize)

    def swapped(packed, scales):
        p = np.asarray(packed, dtype=np.uint8)
        return mxfp4.dequantize(((p & 0xF) << 4) | (p >> 4), scales)

    def scale_per_byte(packed, scales):
        codes = mxfp4.unpack(packed)
        K = codes.shape[-1]
        s = np.asarray(scales, dtype=np.uint8)
        idx = np.minimum(np.arange(K) // 2 // 32 * 2, s.shape[-1] - 1)   # K/2 bytes per 32 * 2
        return oracle.E2M1[codes] * oracle.UE8M0[s[..., idx]]

    assert not _scalar_loop_agrees(swapped)
    assert not _scalar_loop_agrees(scale_per_byte)
