"""The allocation-free layer call, moe_decode_layer_noalloc.

Some callers cannot call cudaMalloc (they run inside another framework's
memory pool, in a plugin's enqueue function, or in a loop that must not block
on an allocation). For them the library offers one layer call that takes no
handle and keeps its intermediate h in static device memory. These tests call
it through the C ABI and check it against moe_decode_layer on the same
inputs, several times in a row (each call finds the previous call's leftovers
in the shared array), with several tokens (two kernels) and with one token
(the one-launch kernel and its counters). This file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_within, bf16_tensor, device_weights, tensor_to_f64, tol_y


def _cfg(E, k, H, I, flags=0):
    from sparse_expert_gemv_gb300 import MoEConfig
    return MoEConfig(E, k, H, I, 0, flags)


def _p(v):
    return ctypes.c_void_p(v)


def test_noalloc_rejects_oversize_and_bad_arguments_on_the_host():
    from sparse_expert_gemv_gb300._lib import MOE_NOALLOC_SCRATCH_BYTES, lib
    z = _p(0)
    w = [_p(256), _p(512), _p(1024), _p(2048)]
    # T * k * I * 2 bytes of h just above the fixed array: refused before any CUDA call
    E, k, H, I = 16, 8, 256, 2048
    T = MOE_NOALLOC_SCRATCH_BYTES // (k * I * 2) + 1
    cfg = _cfg(E, k, H, I)
    assert lib.moe_decode_layer_noalloc(ctypes.byref(cfg), *w, T, z, z, z, z, z) == 2
    assert lib.moe_decode_layer_noalloc(None, *w, 1, z, z, z, z, z) == 1
    assert lib.moe_decode_layer_noalloc(ctypes.byref(_cfg(8, 2, 48, 128)), *w, 1, z, z, z, z, z) == 2
    assert lib.moe_decode_layer_noalloc(ctypes.byref(_cfg(8, 2, 256, 128)), *w, -1, z, z, z, z, z) == 1
    assert lib.moe_decode_layer_noalloc(ctypes.byref(_cfg(8, 2, 256, 128)), _p(256 + 16), *w[1:], 1,
                                        z, z, z, z, z) == 3


@pytest.mark.gpu
def test_noalloc_layer_matches_layer_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_expert_gemv_gb300 import MoEDecode, lib
    dev = torch.device("cuda:0")
    E, k, H, I = 16, 4, 512, 256
    w = wl.Workload(95, "noalloc", E, k, H, I, 6, 0.05)
    experts = wl.make_experts(w, 95, range(E))
    wts = device_weights(w, experts, dev)
    ref_layer = MoEDecode(*wts, k=k, max_T=6)
    # with one token this shape runs as the one-launch kernel, whose CTAs wait
    # for one another on counters in the static array
    assert ref_layer.fused_single_token
    cfg = _cfg(E, k, H, I)
    stream = torch.cuda.current_stream()
    for call, (T, seed) in enumerate([(6, 1), (1, 3), (3, 2), (1, 4)]):
        x = bf16_tensor(wl.make_x(w, seed, T), dev)
        ids_np, tw_np = oracle.route(wl.make_logits(w, seed, T), k)
        ids = torch.from_numpy(ids_np).to(dev)
        tw = torch.from_numpy(tw_np).to(dev)
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=dev)
        st = lib.moe_decode_layer_noalloc(ctypes.byref(cfg), *[_p(t.data_ptr()) for t in wts], T,
                                          _p(x.data_ptr()), _p(ids.data_ptr()), _p(tw.data_ptr()),
                                          _p(y.data_ptr()), _p(stream.cuda_stream))
        assert st == 0, f"call {call}: status {st}"
        y_ref = ref_layer.layer(x, ids, tw)
        torch.cuda.synchronize()
        ref = tensor_to_f64(y_ref)
        assert_within(tensor_to_f64(y), ref, tol_y(ref), f"noalloc call {call}")
    ref_layer.close()
