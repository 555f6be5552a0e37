"""ctypes view of libmoe_decode.so (the C ABI declared in include/moe_decode.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Importing this module fails loudly when the library has not been
built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_decode.so")

MOE_OK = 0
MOE_DEVICE_BAD_ID = 0x1
MOE_DEVICE_TIMEOUT = 0x2
MOE_FLAG_NO_PDL = 0x1
MOE_FLAG_HOST_COPY = 0x2
MOE_FLAG_MXFP4 = 0x4
MOE_FLAG_WARP_MMA = 0x8
MOE_PATH_AUTO = 0
MOE_PATH_WARP = 1
MOE_PATH_TENSOR = 2
MOE_NOALLOC_SCRATCH_BYTES = 1 << 20

STATUS_NAMES = {
    0: "MOE_OK",
    1: "MOE_ERR_INVALID_ARG",
    2: "MOE_ERR_UNSUPPORTED_SHAPE",
    3: "MOE_ERR_MISALIGNED",
    4: "MOE_ERR_CUDA",
    5: "MOE_ERR_DEVICE_FAULT",
}


class MoEConfig(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("k", ctypes.c_int32), ("H", ctypes.c_int32),
                ("I", ctypes.c_int32), ("max_T", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}" if what else
                         STATUS_NAMES.get(status, str(status)))


class MoEPlan(ctypes.Structure):
    """moe_decode_plan_t: the launch plan moe_decode_plan reports."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "fused", "fused_kc", "fused_slots", "fused_slot_bytes", "fused_down_rows",
        "fused_down_per_slot", "fused_smem", "gate_up_group", "gate_up_kernel", "gate_up_slots",
        "gate_up_smem", "down_kernel", "down_slots", "down_smem")]


_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_st = ctypes.c_int

# name -> (restype, argtypes); one line per entry point of include/moe_decode.h
SIGNATURES = {
    "moe_decode_create": (_st, [ctypes.POINTER(MoEConfig), _p, _p, _p, _p, ctypes.POINTER(_p)]),
    "moe_decode_destroy": (_st, [_p]),
    "moe_route": (_st, [_p, _i32, _p, _p, _p, _p]),
    "moe_dedup_schedule": (_st, [_p, _i32, _p, _p, _p, _p, _p, _p]),
    "moe_gate_up": (_st, [_p, _i32, _p, _p, _p, _p]),
    "moe_down": (_st, [_p, _i32, _p, _p, _p, _p, _p]),
    "moe_decode_layer": (_st, [_p, _i32, _p, _p, _p, _p, _p, _p]),
    "moe_decode_forward_host": (_st, [_p, _i32, _p, _p, _p, _p, _p]),
    "moe_decode_get_error": (_st, [_p, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_decode_get_error_stream": (_st, [_p, _p, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_status_string": (ctypes.c_char_p, [_st]),
    "moe_decode_version": (_i32, []),
    "moe_decode_fused_layer": (_i32, [_p]),
    "moe_decode_set_path": (_st, [_p, _i32]),
    "moe_decode_path": (_i32, [_p, _i32]),
    "moe_decode_tensor_path": (_i32, [_p]),
    "moe_decode_kernel_name": (ctypes.c_char_p, [_p, _i32, _i32]),
    "moe_decode_plan": (_st, [ctypes.POINTER(MoEConfig), _i32, _i32, _i32, ctypes.POINTER(MoEPlan)]),
    "moe_decode_arm_barrier_timeout": (_st, [_p]),
    "moe_decode_layer_noalloc": (_st, [ctypes.POINTER(MoEConfig), _p, _p, _p, _p, _i32, _p, _p, _p,
                                       _p, _p]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = load()


def check(status: int, what: str = "") -> None:
    if status != MOE_OK:
        raise MoEError(status, what)
