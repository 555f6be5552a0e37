"""Output-centric small-batch MoE decode layer for GB300 (sm_103a).

The layer of the warp-decode post (cursor.com/blog/warp-decode): tokens are
routed to k of E experts; a gate/up kernel computes SiLU(gate) * up per
(token, routed expert, neuron) and a down kernel computes the routing-weighted
sum over the top-k experts per (token, output dimension). Weights are MXFP8
(E4M3 codes with one UE8M0 scale per 32 elements along the reduction axis),
decoded to FP32 in registers, one warp per output.

The compute lives in libmoe_decode.so (C ABI, include/moe_decode.h). This
package is a thin ctypes binding: PyTorch supplies device memory and streams.
"""
from ._lib import (LIB_PATH, MOE_DEVICE_BAD_ID, MOE_DEVICE_TIMEOUT, MOE_FLAG_HOST_COPY,
                   MOE_FLAG_MXFP4, MOE_FLAG_NO_PDL, MOE_FLAG_WARP_MMA, MoEConfig, MoEError, check,
                   lib)
from .layer import MoEDecode

__all__ = ["MoEDecode", "MoEError", "MoEConfig", "lib", "check", "LIB_PATH",
           "MOE_DEVICE_BAD_ID", "MOE_DEVICE_TIMEOUT", "MOE_FLAG_HOST_COPY", "MOE_FLAG_MXFP4",
           "MOE_FLAG_NO_PDL", "MOE_FLAG_WARP_MMA"]
