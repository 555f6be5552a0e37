"""Python face of one MoE decode layer: a handle plus the C ABI's calls.

Every method forwards device pointers of torch tensors and the current CUDA
stream to libmoe_decode.so; nothing is computed here.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import (MOE_FLAG_MXFP4, MOE_PATH_AUTO, MOE_PATH_TENSOR, MOE_PATH_WARP, MoEConfig, check,
                   lib)


def _ptr(t: torch.Tensor | None) -> int:
    # a plain int: the entry points' argtypes make it a void*
    return 0 if t is None else t.data_ptr()


def _stream(stream: torch.cuda.Stream | None) -> int:
    if stream is not None:
        return stream.cuda_stream
    # the current stream's handle, without building a Stream object per call
    # where torch offers that
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _need(t: torch.Tensor, dtype: torch.dtype, shape: tuple, name: str, cuda: bool = True) -> None:
    # one cheap test on the common path; the detailed ones only on failure
    if (isinstance(t, torch.Tensor) and t.dtype is dtype and t.shape == shape
            and t.is_cuda is cuda and t.is_contiguous()):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    raise ValueError(f"{name} must be a host tensor")


class MoEDecode:
    """One MoE decode layer over caller-owned block-scaled weights on the current device.

    fmt="mxfp8": w_gateup uint8 [E, 2I, H] (rows [0, I) gate, [I, 2I) up),
    w_down uint8 [E, H, I], one E4M3 code per byte. fmt="mxfp4": w_gateup
    uint8 [E, 2I, H/2], w_down uint8 [E, H, I/2], two E2M1 codes per byte
    (the even element in the low nibble). Either way s_gateup uint8
    [E, 2I, H/32] and s_down uint8 [E, H, I/32] hold the UE8M0 scales. The
    tensors are borrowed (kept alive by this object, never copied).
    """

    def __init__(self, w_gateup, s_gateup, w_down, s_down, *, k: int, max_T: int = 32,
                 flags: int = 0, fmt: str = "mxfp8"):
        if fmt not in ("mxfp8", "mxfp4"):
            raise ValueError(f"fmt must be 'mxfp8' or 'mxfp4', got {fmt!r}")
        per = 2 if fmt == "mxfp4" else 1          # elements per code byte
        E, twoI, RB = w_gateup.shape
        I, H = twoI // 2, RB * per
        _need(w_gateup, torch.uint8, (E, 2 * I, H // per), "w_gateup")
        _need(s_gateup, torch.uint8, (E, 2 * I, H // 32), "s_gateup")
        _need(w_down, torch.uint8, (E, H, I // per), "w_down")
        _need(s_down, torch.uint8, (E, H, I // 32), "s_down")
        self.E, self.k, self.H, self.I, self.max_T, self.fmt = E, k, H, I, max_T, fmt
        self._weights = (w_gateup, s_gateup, w_down, s_down)
        if fmt == "mxfp4":
            flags |= MOE_FLAG_MXFP4
        cfg = MoEConfig(E, k, H, I, max_T, flags)
        h = ctypes.c_void_p()
        check(lib.moe_decode_create(ctypes.byref(cfg), _ptr(w_gateup), _ptr(s_gateup),
                                    _ptr(w_down), _ptr(s_down), ctypes.byref(h)),
              "moe_decode_create")
        self._h = h

    # -- lifetime -------------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "_h", None):
            lib.moe_decode_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    @property
    def fused_single_token(self) -> bool:
        """True when one-token layer calls run as one persistent launch."""
        return lib.moe_decode_fused_layer(self._h) == 1

    @property
    def tensor_path(self) -> bool:
        """True when this handle can run the expert-centric tensor-core path."""
        return lib.moe_decode_tensor_path(self._h) == 1

    def set_path(self, path: str) -> None:
        """Which form layer calls take: "auto" (the tensor-core path from 16
        tokens when they route 1.5 or more slots per expert on average),
        "warp" or "tensor"."""
        code = {"auto": MOE_PATH_AUTO, "warp": MOE_PATH_WARP, "tensor": MOE_PATH_TENSOR}[path]
        check(lib.moe_decode_set_path(self._h, code), "moe_decode_set_path")

    def path(self, T: int) -> str:
        """The form a layer call with T tokens takes: "warp" or "tensor"."""
        return {MOE_PATH_WARP: "warp", MOE_PATH_TENSOR: "tensor"}[lib.moe_decode_path(self._h, T)]

    def kernel_name(self, T: int, which: str) -> str:
        """The kernel moe_gate_up (which="gate_up") or moe_down ("down")
        launches for T tokens on this handle."""
        w = {"gate_up": 0, "down": 1}[which]
        return lib.moe_decode_kernel_name(self._h, T, w).decode()

    def arm_barrier_timeout(self) -> None:
        """Test support: the next one-launch call's grid barrier times out
        (bounded; it sets MOE_DEVICE_TIMEOUT, which get_error reports)."""
        check(lib.moe_decode_arm_barrier_timeout(self._h), "moe_decode_arm_barrier_timeout")

    def _dev(self, shape, dtype, out, name):
        if out is None:
            return torch.empty(shape, dtype=dtype, device=self._weights[0].device)
        _need(out, dtype, shape, name)
        return out

    # -- calls ----------------------------------------------------------------
    def route(self, logits, ids=None, w=None, stream=None):
        T = logits.shape[0]
        _need(logits, torch.float32, (T, self.E), "logits")
        ids = self._dev((T, self.k), torch.int32, ids, "topk_ids")
        w = self._dev((T, self.k), torch.float32, w, "topk_w")
        check(lib.moe_route(self._h, T, _ptr(logits), _ptr(ids), _ptr(w), _stream(stream)),
              "moe_route")
        return ids, w

    def dedup_schedule(self, ids, stream=None):
        T = ids.shape[0]
        _need(ids, torch.int32, (T, self.k), "topk_ids")
        U = min(self.E, T * self.k)
        dev = ids.device
        uniq = torch.full((U,), -1, dtype=torch.int32, device=dev)
        off = torch.full((U + 1,), -1, dtype=torch.int32, device=dev)
        pairs = torch.full((T * self.k,), -1, dtype=torch.int32, device=dev)
        n = torch.zeros((1,), dtype=torch.int32, device=dev)
        check(lib.moe_dedup_schedule(self._h, T, _ptr(ids), _ptr(uniq), _ptr(off), _ptr(pairs),
                                     _ptr(n), _stream(stream)), "moe_dedup_schedule")
        return uniq, off, pairs, n

    def gate_up(self, x, ids, h=None, stream=None):
        T = x.shape[0]
        _need(x, torch.bfloat16, (T, self.H), "x")
        _need(ids, torch.int32, (T, self.k), "topk_ids")
        h = self._dev((T, self.k, self.I), torch.bfloat16, h, "h")
        check(lib.moe_gate_up(self._h, T, _ptr(x), _ptr(ids), _ptr(h), _stream(stream)),
              "moe_gate_up")
        return h

    def down(self, h, ids, w, y=None, stream=None):
        T = h.shape[0]
        _need(h, torch.bfloat16, (T, self.k, self.I), "h")
        _need(ids, torch.int32, (T, self.k), "topk_ids")
        _need(w, torch.float32, (T, self.k), "topk_w")
        y = self._dev((T, self.H), torch.bfloat16, y, "y")
        check(lib.moe_down(self._h, T, _ptr(h), _ptr(ids), _ptr(w), _ptr(y), _stream(stream)),
              "moe_down")
        return y

    def layer(self, x, ids, w, h=None, y=None, stream=None):
        T = x.shape[0]
        _need(x, torch.bfloat16, (T, self.H), "x")
        _need(ids, torch.int32, (T, self.k), "topk_ids")
        _need(w, torch.float32, (T, self.k), "topk_w")
        h = self._dev((T, self.k, self.I), torch.bfloat16, h, "h")
        y = self._dev((T, self.H), torch.bfloat16, y, "y")
        check(lib.moe_decode_layer(self._h, T, _ptr(x), _ptr(ids), _ptr(w), _ptr(h), _ptr(y),
                                   _stream(stream)), "moe_decode_layer")
        return y

    def forward_host(self, x, ids, w, y=None, stream=None):
        """The layer from and to host tensors (pin them for asynchronous copies)."""
        T = x.shape[0]
        _need(x, torch.bfloat16, (T, self.H), "x", cuda=False)
        _need(ids, torch.int32, (T, self.k), "topk_ids", cuda=False)
        _need(w, torch.float32, (T, self.k), "topk_w", cuda=False)
        if y is None:
            y = torch.empty((T, self.H), dtype=torch.bfloat16, pin_memory=True)
        _need(y, torch.bfloat16, (T, self.H), "y", cuda=False)
        check(lib.moe_decode_forward_host(self._h, T, _ptr(x), _ptr(ids), _ptr(w), _ptr(y),
                                          _stream(stream)), "moe_decode_forward_host")
        return y

    def get_error(self, stream=None) -> int:
        """Read and clear the handle's device error bits. Waits for this
        handle's latest call, or, given a stream, for that stream."""
        flags = ctypes.c_uint32(0)
        if stream is None:
            st = lib.moe_decode_get_error(self._h, ctypes.byref(flags))
        else:
            st = lib.moe_decode_get_error_stream(self._h, _stream(stream), ctypes.byref(flags))
        if st not in (0, 5):
            check(st, "moe_decode_get_error")
        return int(flags.value)
