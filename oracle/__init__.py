"""CPU oracle for the small-batch MoE decode layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this package: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg use it. It shares no code with the CUDA library
(no kernels, headers, tables or helpers); the only module both sides use is
`workloads`, which draws and encodes the seeded inputs.

Everything here is plain numpy in float64, written from the definitions on the
pages (cited per function):

  mxfp8    E4M3 and UE8M0 decode tables and block dequantisation
  mxfp4    E2M1 decode table, nibble unpacking and block dequantisation
  bf16     round-to-nearest-even from float64 to bfloat16 values
  moe      routing, the dedup schedule, the gate/up and down projections

Pins (tests/test_oracle_*.py) tie each function to something other than
itself: torch's float8 and bfloat16 conversions, exhaustive bit-pattern
sweeps, brute-force scalar loops, a dense special case against numpy matmul,
and invariants of the layer.
"""
from .mxfp8 import E4M3, UE8M0, e4m3_decode, ue8m0_decode, dequantize
from .mxfp4 import E2M1, e2m1_decode
from .mxfp4 import dequantize as dequantize_mxfp4
from .bf16 import bf16_rne
from .moe import (silu, route, dedup_schedule, gate_up, down, layer,
                  requantize_mxfp8, layer_classic)

__all__ = [
    "E4M3", "UE8M0", "e4m3_decode", "ue8m0_decode", "dequantize", "bf16_rne",
    "E2M1", "e2m1_decode", "dequantize_mxfp4",
    "silu", "route", "dedup_schedule", "gate_up", "down", "layer",
    "requantize_mxfp8", "layer_classic",
]
