"""Round-to-nearest-even from float64 straight to bfloat16 values.

The warp-decode post (cursor.com/blog/warp-decode), "Improved accuracy", keeps
activations in BF16 with FP32 accumulators; the intermediate h and the output y
are therefore stored as BF16. The oracle mirrors that storage rounding.

bfloat16 keeps 8 significant bits (1 implicit + 7 stored) with float32's
exponent range: normal numbers down to 2^-126, subnormals in steps of 2^-133,
largest finite (2 - 2^-7) * 2^127. Rounding goes directly from float64: rounding
to float32 first and then to bf16 would round twice, which is wrong for values
just off a bf16 midpoint.
"""
from __future__ import annotations

import numpy as np

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_rne(a) -> np.ndarray:
    """float64 array -> float64 array of the nearest bf16 values (ties to even)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.array(a, copy=True)
    fin = np.isfinite(a) & (a != 0)
    v = a[fin]
    _, ex = np.frexp(v)                       # |v| = m * 2^ex, m in [0.5, 1)
    # quantum: 2^(ex-8) for normals (8 significant bits), 2^-133 below 2^-126
    q_exp = np.maximum(ex, -125) - 8
    r = np.ldexp(np.rint(np.ldexp(v, -q_exp)), q_exp)   # np.rint rounds half to even
    big = np.abs(r) > _BF16_MAX
    r[big] = np.copysign(np.inf, r[big])
    out[fin] = r
    return out
