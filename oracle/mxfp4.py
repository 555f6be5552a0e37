"""MXFP4 decode: E2M1 element codes, two to a byte, one UE8M0 scale per 32 elements.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Format source: the GC-MoE summary (onedev.kr/papers/1690), section "How it is
used": on its Blackwell path the routed expert weights are FP4 E2M1 with the
same K32 granularity as the activations' UE8M0 scales. The page gives no bit
layouts; the reading used here is the OCP MX definition of E2M1:

  E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. Exponent
      field 0 is subnormal: (m/2) * 2^0. Otherwise (1 + m/2) * 2^(e-1).
      There is no infinity and no NaN: the largest magnitude is 6 (0x7).
  UE8M0: as for MXFP8 (oracle.mxfp8), 2^(s-127), 0xFF is NaN.

Packing (the page is silent; reading): a row of K elements is K/2 bytes;
element 2c sits in the low nibble of byte c and element 2c+1 in its high
nibble. Scales stay one byte per 32 elements of the row.

Dequantisation is a table lookup, exact in float64:
  dq(W)[r, K] = E2M1[nibble(W, r, K)] * UE8M0[S[r, K // 32]].
"""
from __future__ import annotations

import numpy as np

from .mxfp8 import UE8M0

BLOCK = 32


def e2m1_decode(code: int) -> float:
    """Value of one 4-bit E2M1 code from its sign, exponent and mantissa fields."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * (m / 2.0)
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1 = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)
E2M1.setflags(write=False)


def unpack(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> 4-bit codes uint8 [..., K] (low nibble first)."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def dequantize(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """dq(W): float64 [..., K] from packed E2M1 codes [..., K/2] and UE8M0 scales [..., K/32]."""
    codes = unpack(packed)
    scales = np.asarray(scales, dtype=np.uint8)
    K = codes.shape[-1]
    if K % BLOCK or scales.shape[-1] != K // BLOCK or scales.shape[:-1] != codes.shape[:-1]:
        raise ValueError(f"shape mismatch: packed {np.shape(packed)} scales {scales.shape}")
    vals = E2M1[codes]
    s = UE8M0[scales]
    return (vals.reshape(*codes.shape[:-1], K // BLOCK, BLOCK) * s[..., None]).reshape(codes.shape)
