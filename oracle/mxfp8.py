"""MXFP8 decode: E4M3 element codes with one UE8M0 scale per 32 elements.

Format source: the GC-MoE summary (onedev.kr/papers/1690), section "How it is
used", names the Blackwell block format: FP8 E4M3 values with one UE8M0 scale
per 32 values along K. The warp-decode post (cursor.com/blog/warp-decode),
"How the two kernels work", converts such MXFP8 weights to FP32 on the fly.
Neither page spells out the bit layouts; the reading used here is the OCP MX
definition of the two element types:

  E4M3 (the "FN" flavour MX uses): 1 sign bit, 4 exponent bits (bias 7),
      3 mantissa bits. Exponent field 0 is subnormal: (m/8) * 2^-6.
      Otherwise (1 + m/8) * 2^(e-7). There is no infinity; S.1111.111 is NaN,
      so the largest magnitude is 448 (0x7E).
  UE8M0: an 8-bit unsigned exponent, value 2^(s-127); 0xFF is NaN.

The tables are built from those bit fields; dequantisation is a table lookup
(dq(W)[r, K] = E4M3[W[r, K]] * UE8M0[S[r, K // 32]]), exact in float64.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK = 32


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code from its sign, exponent and mantissa fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def ue8m0_decode(code: int) -> float:
    """Value of one UE8M0 scale code: 2^(code-127), NaN for 0xFF."""
    code = int(code) & 0xFF
    if code == 0xFF:
        return math.nan
    return math.ldexp(1.0, code - 127)


E4M3 = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
E4M3.setflags(write=False)
UE8M0 = np.array([ue8m0_decode(c) for c in range(256)], dtype=np.float64)
UE8M0.setflags(write=False)


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """dq(W): float64 [..., K] from E4M3 codes [..., K] and UE8M0 scales [..., K/32]."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    K = codes.shape[-1]
    if K % BLOCK or scales.shape[-1] != K // BLOCK or scales.shape[:-1] != codes.shape[:-1]:
        raise ValueError(f"shape mismatch: codes {codes.shape} scales {scales.shape}")
    vals = E4M3[codes]
    s = UE8M0[scales]
    return (vals.reshape(*codes.shape[:-1], K // BLOCK, BLOCK) * s[..., None]).reshape(codes.shape)
