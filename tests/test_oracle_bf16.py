"""Pins for the oracle's float64 -> bf16 round-to-nearest-even."""
import numpy as np
import torch

import oracle


def all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    return bits, v


def test_every_bf16_value_is_a_fixed_point():
    _, v = all_bf16_values()
    fin = np.isfinite(v)
    got = oracle.bf16_rne(v[fin])
    assert np.array_equal(got, v[fin])
    assert np.array_equal(np.signbit(got), np.signbit(v[fin]))
    inf = np.isinf(v)
    assert np.array_equal(oracle.bf16_rne(v[inf]), v[inf])
    assert np.all(np.isnan(oracle.bf16_rne(v[np.isnan(v)])))


def test_midpoints_round_to_even_pattern():
    # between two consecutive finite positive bf16 patterns b and b+1 the exact
    # midpoint must go to the one whose last stored bit is 0
    bits, v = all_bf16_values()
    lo_bits = np.concatenate([np.arange(0, 0x7F7F), np.arange(0x8000, 0xFF7F)])
    a, b = v[lo_bits], v[lo_bits + 1]
    mid = (a + b) / 2.0                # exact in float64
    want = np.where(lo_bits % 2 == 0, a, b)
    got = oracle.bf16_rne(mid)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [hex(x) for x in lo_bits[bad[:5]]]


def test_random_float32_matches_torch():
    rng = np.random.default_rng(3)
    a = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(50000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(50000) * 1e37).astype(np.float32),
        rng.integers(0, 2**32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    a = a[np.isfinite(a)]
    want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_rne(a.astype(np.float64))
    assert np.array_equal(got, want)


def test_direct_rounding_not_double_rounding():
    # x = 1 + 2^-8 + 2^-40 lies just above the bf16 midpoint between 1 and
    # 1 + 2^-7. Correct rounding gives 1 + 2^-7; rounding through float32
    # first lands exactly on the midpoint and then ties down to 1.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_rne(np.array([x]))[0] == 1.0 + 2.0 ** -7
    assert oracle.bf16_rne(np.array([-x]))[0] == -(1.0 + 2.0 ** -7)
    via_f32 = torch.tensor([x], dtype=torch.float64).to(torch.float32).to(torch.bfloat16).item()
    assert via_f32 == 1.0


def test_overflow_and_underflow():
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    half_ulp = 2.0 ** 119
    assert oracle.bf16_rne(np.array([big]))[0] == big
    assert oracle.bf16_rne(np.array([big + half_ulp * 0.99]))[0] == big
    assert np.isinf(oracle.bf16_rne(np.array([big + half_ulp]))[0])
    tiny = 2.0 ** -133
    assert oracle.bf16_rne(np.array([tiny]))[0] == tiny
    assert oracle.bf16_rne(np.array([tiny * 0.5]))[0] == 0.0          # tie to even (zero)
    assert oracle.bf16_rne(np.array([tiny * 0.51]))[0] == tiny
    assert oracle.bf16_rne(np.array([tiny * 1.5]))[0] == 2 * tiny     # tie to even
