"""Seeded synthetic inputs for the small-batch MoE decode layer.

This module is shared by the CPU oracle's tests, the CUDA parity tests and the
benchmark. It holds no arithmetic of the layer itself (no MXFP8 decode, no
projections, no routing): it only draws random numbers and encodes them into
the storage formats the layer consumes.

Workloads (the five decode shapes the layer is specified on):

  0  tiny layer      E=8   k=2 H=256  I=128  T=1   sigma=0.02
  1  batch-1 decode  E=128 k=8 H=2048 I=768  T=1   sigma=0.02
  2  small batch     E=128 k=8 H=2048 I=768  T=8   sigma=0.02
  3  skewed routing  E=128 k=8 H=2048 I=768  T=32  sigma=0.02, Zipf(1.1) router prior
  4  large experts   E=256 k=8 H=7168 I=2048 T=16  sigma=0.01

Recipe (seed_c = 1000 + c; every stream is numpy's PCG64 seeded with the
integer list [seed, stream, index], so any expert can be regenerated alone):

  x       stream 1: N(0,1) float32, rounded to bf16 (round-to-nearest-even)
  logits  stream 2: N(0,1) float32; workload 3 adds log p_e with
          p_e ~ r_e^-1.1, r_e = 1 + perm[e], perm from stream 5, so the hot
          experts sit at scattered addresses
  W_gateup[e] stream 3 index e: N(0, sigma) float32 [2I, H], rows [0, I) are
          the gate projection and rows [I, 2I) the up projection
  W_down[e]   stream 4 index e: N(0, sigma) float32 [H, I]

Weights are stored as MXFP8: one E4M3 code per element and one UE8M0 scale
code per 32 consecutive elements along the reduction axis (the block format
the GC-MoE summary, onedev.kr/papers/1690, "How it is used", names for
Blackwell activations). The encoder follows the usual MX recipe: per 32-block
shared exponent = floor(log2(amax)) - 8 clamped to [-127, 127] (scale code =
exponent + 127; an all-zero block gets code 127), elements divided by 2^exp,
saturated to +-448 and rounded to the nearest E4M3 value (ties to even). It
never emits a NaN code.

The MXFP4 variant of every workload draws the same float weights and stores
them as E2M1 codes, two to a byte (element 2c in the low nibble of byte c,
element 2c+1 in the high nibble), with the same UE8M0 scale layout (the
routed-weight format the GC-MoE summary, "How it is used", names for
Blackwell). Its encoder follows the same MX recipe with E2M1's largest
exponent: shared exponent = floor(log2(amax)) - 2, elements divided by 2^exp,
saturated to +-6 and rounded to the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6
(ties to the even code); the sign bit follows the element's sign, so small
negative elements become -0.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

__all__ = [
    "Workload", "WORKLOADS", "workload", "seed_of",
    "make_x", "make_logits", "encode_mxfp8", "encode_mxfp4", "make_expert", "make_experts",
    "make_expert_float",
    "FORMATS",
    "bf16_bits_to_f64", "NAN_CODE",
]

# E4M3 code 0x7F is NaN; used to fill experts a test must never read.
NAN_CODE = 0x7F


@dataclasses.dataclass(frozen=True)
class Workload:
    idx: int
    name: str
    E: int
    k: int
    H: int
    I: int
    T: int
    sigma: float
    zipf: float | None = None

    @property
    def weight_bytes_per_expert(self) -> int:
        """E4M3 codes plus UE8M0 scales of one expert's three projections."""
        return self.weight_bytes("mxfp8")

    def weight_bytes(self, fmt: str = "mxfp8") -> int:
        """Codes plus UE8M0 scales of one expert's three projections in `fmt`."""
        codes = 3 * self.H * self.I
        return (codes if fmt == "mxfp8" else codes // 2) + codes // 32


WORKLOADS = {
    0: Workload(0, "tiny E8 k2 H256 I128 T1", 8, 2, 256, 128, 1, 0.02),
    1: Workload(1, "batch-1 decode E128 k8 H2048 I768 T1", 128, 8, 2048, 768, 1, 0.02),
    2: Workload(2, "small-batch decode E128 k8 H2048 I768 T8", 128, 8, 2048, 768, 8, 0.02),
    3: Workload(3, "skewed-routing decode E128 k8 H2048 I768 T32 zipf1.1", 128, 8, 2048, 768, 32, 0.02, 1.1),
    4: Workload(4, "large-expert decode E256 k8 H7168 I2048 T16", 256, 8, 7168, 2048, 16, 0.01),
}


def workload(c: int) -> Workload:
    return WORKLOADS[c]


def seed_of(c: int) -> int:
    return 1000 + c


def _rng(seed: int, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, stream, index])


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of bf16 bit patterns (a widening, no rounding)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def make_x(w: Workload, seed: int, T: int | None = None) -> np.ndarray:
    """x[T, H] as bf16 bit patterns (uint16)."""
    T = w.T if T is None else T
    a = _rng(seed, 1).standard_normal((T, w.H), dtype=np.float32)
    return _to_bf16_bits(a)


def make_logits(w: Workload, seed: int, T: int | None = None, step: int = 0) -> np.ndarray:
    """Router logits[T, E] float32 (workload 3 carries the Zipf prior)."""
    T = w.T if T is None else T
    z = _rng(seed, 2, step).standard_normal((T, w.E))
    if w.zipf is not None:
        perm = _rng(seed, 5).permutation(w.E)
        r = 1.0 + perm.astype(np.float64)
        p = r ** (-w.zipf)
        p /= p.sum()
        z = z + np.log(p)[None, :]
    return z.astype(np.float32)


def encode_mxfp8(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """float32 [R, K] (K % 32 == 0) -> (E4M3 codes uint8 [R, K], UE8M0 codes uint8 [R, K/32])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    R, K = w.shape
    assert K % 32 == 0
    b = torch.from_numpy(w).view(R, K // 32, 32)
    amax = b.abs().amax(-1)
    _, ex = torch.frexp(amax)                      # amax = m * 2^ex, m in [0.5, 1)
    e = (ex - 1 - 8).clamp(-127, 127)              # floor(log2 amax) - 8
    e = torch.where(amax == 0, torch.zeros_like(e), e)
    inv = torch.exp2(-e.to(torch.float64)).to(torch.float32)  # exact powers of two
    q = (b * inv[..., None]).clamp(-448.0, 448.0)
    codes = q.reshape(R, K).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    scales = (e + 127).to(torch.uint8).numpy().copy()
    return codes, scales


# magnitudes of the E2M1 codes 0..7, the rounding targets of encode_mxfp4
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def encode_mxfp4(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """float32 [R, K] (K % 32 == 0) -> (packed E2M1 codes uint8 [R, K/2], UE8M0 codes uint8 [R, K/32])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    R, K = w.shape
    assert K % 32 == 0
    b = w.reshape(R, K // 32, 32).astype(np.float64)
    amax = np.abs(b).max(axis=-1)
    _, ex = np.frexp(amax)                         # amax = m * 2^ex, m in [0.5, 1)
    e = np.clip(ex - 1 - 2, -127, 127)             # floor(log2 amax) - 2
    e = np.where(amax == 0, 0, e)
    q = np.ldexp(b, -e[..., None])
    a = np.minimum(np.abs(q), 6.0)
    hi = np.clip(np.searchsorted(_E2M1_GRID, a, side="left"), 0, 7)
    lo = np.clip(hi - 1, 0, 7)
    dlo, dhi = a - _E2M1_GRID[lo], _E2M1_GRID[hi] - a
    mag = np.where((dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0)), hi, lo)
    codes = (mag | (np.signbit(q).astype(np.int64) << 3)).astype(np.uint8).reshape(R, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = (e + 127).astype(np.uint8)
    return packed, scales


FORMATS = {"mxfp8": encode_mxfp8, "mxfp4": encode_mxfp4}


def make_expert_float(w: Workload, seed: int, e: int):
    """One expert's weights as drawn, before any encoding: (W_gateup float32
    [2I, H], None, W_down float32 [H, I], None) (the full-precision weights the
    encoded ones approximate)."""
    gu = _rng(seed, 3, e).standard_normal((2 * w.I, w.H), dtype=np.float32)
    gu *= np.float32(w.sigma)
    dn = _rng(seed, 4, e).standard_normal((w.H, w.I), dtype=np.float32)
    dn *= np.float32(w.sigma)
    return gu, None, dn, None


def make_expert(w: Workload, seed: int, e: int, fmt: str = "mxfp8"):
    """One expert's weight tensors in `fmt` ("mxfp8" or "mxfp4"):
    (wgu [2I, H*c], sgu [2I, H/32], wd [H, I*c], sd [H, I/32]), c = 1 code
    byte per element for MXFP8 and 1/2 for MXFP4."""
    enc = FORMATS[fmt]
    gu = _rng(seed, 3, e).standard_normal((2 * w.I, w.H), dtype=np.float32)
    gu *= np.float32(w.sigma)
    wgu, sgu = enc(gu)
    del gu
    dn = _rng(seed, 4, e).standard_normal((w.H, w.I), dtype=np.float32)
    dn *= np.float32(w.sigma)
    wd, sd = enc(dn)
    return wgu, sgu, wd, sd


def make_experts(w: Workload, seed: int, experts, threads: int | None = None,
                 fmt: str = "mxfp8") -> dict:
    """{e: make_expert(w, seed, e, fmt)} for the given expert ids, generated in parallel."""
    experts = sorted(set(int(e) for e in experts))
    threads = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        out = list(ex.map(lambda e: make_expert(w, seed, e, fmt), experts))
    return dict(zip(experts, out))
