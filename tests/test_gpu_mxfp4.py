"""GPU parity of the MXFP4 weight format (E2M1 codes two to a byte, UE8M0
scales per 32) against the float64 oracle, with the tolerances of
test_gpu_parity (one bf16 step of h and y plus 1e-3 rms): the seeded
workloads, ragged and degenerate shapes, the one-launch single-token form,
duplicate and invalid ids, and the host and allocation-free entry points."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import (Case, assert_within, bf16_tensor, check_layer_call, device_weights, metrics, tensor_to_f64,
                      tol_h, tol_y)
from test_gpu_edges import Small, _layer_once

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _check_case(case: Case, dev, expect_fused=None):
    from sparse_expert_gemv_gb300 import MoEDecode
    w = case.w
    layer = MoEDecode(*device_weights(w, case.experts, dev, fmt="mxfp4"), k=w.k,
                      max_T=max(case.T, 1), fmt="mxfp4")
    if expect_fused is not None:
        assert layer.fused_single_token == expect_fused
    x = bf16_tensor(case.x_bits, dev)
    ids = torch.from_numpy(case.ids).to(dev)
    tw = torch.from_numpy(case.tw).to(dev)
    h = layer.gate_up(x, ids)
    y = layer.down(h, ids, tw)
    torch.cuda.synchronize()
    ref = case.ref()
    S = case.tokens
    hm = assert_within(tensor_to_f64(h)[S], ref["h_spec"][S], tol_h(ref["h_spec"][S]), "h")
    ym = assert_within(tensor_to_f64(y)[S], ref["y_spec"][S], tol_y(ref["y_spec"][S]), "y")
    check_layer_call(layer, case, x, ids, tw, y, fmt="mxfp4")
    assert layer.get_error() == 0
    layer.close()
    return hm, ym, metrics(tensor_to_f64(y)[S], ref["y_pure"][S])


@pytest.mark.parametrize("c", [0, 1, 2, 3])
def test_mxfp4_workload_parity_full(c, dev):
    hm, ym, pure = _check_case(Case(c, fmt="mxfp4"), dev, expect_fused={0: False, 1: True}.get(c))
    print(f"mxfp4 workload {c}: h {hm}  y {ym}  y vs fp64-exact {pure}")
    assert ym["cosine"] > 0.9999


def test_mxfp4_workload4_sampled_tokens(dev):
    # E=256, H=7168, I=2048, T=16 over a full 5.9 GB MXFP4 weight set (the 16
    # tokens' x does not fit shared memory, so gate/up runs as two launches of
    # 8 tokens whose x is staged); three tokens' experts hold real weights,
    # every other expert NaN scales
    hm, ym, _ = _check_case(Case(4, tokens=[0, 7, 15], fmt="mxfp4"), dev)
    print(f"mxfp4 workload 4 (tokens 0,7,15): h {hm}  y {ym}")


@pytest.mark.parametrize("E,k,H,I,T", [
    (5, 3, 1184, 96, 5),      # 37 blocks per row: ragged lanes; k odd
    (16, 16, 64, 64, 3),      # k > 8
    (8, 2, 256, 128, 37),     # T > 32: two token groups
    (3, 1, 32, 32, 1),        # smallest shapes (one 16-byte block per row)
    (64, 8, 2048, 32, 6),     # I = 32
    (4, 4, 96, 160, 33),      # every expert shared by many tokens, 2 groups
    (8, 2, 512, 128, 1),      # T = 1 below the one-launch minimum H for MXFP4
])
def test_mxfp4_ragged_shapes(dev, E, k, H, I, T):
    s = Small(dev, E, k, H, I, T, fmt="mxfp4")
    s.check()
    assert s.layer.get_error() == 0


@pytest.mark.parametrize("E,k,H,I", [(16, 4, 1024, 256), (64, 8, 2048, 768),
                                     (12, 8, 7168, 2048), (6, 5, 3072, 384), (8, 2, 1024, 128)])
def test_mxfp4_single_token_layer(dev, E, k, H, I):
    s = Small(dev, E, k, H, I, 1, seed=E + H, fmt="mxfp4")
    assert s.layer.fused_single_token
    h, y = _layer_once(s)
    r = s.ref()
    assert_within(tensor_to_f64(h), r["h_spec"], tol_h(r["h_spec"]), "h")
    assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y")
    _, y2 = s.run()
    assert_within(tensor_to_f64(y2), r["y_spec"], tol_y(r["y_spec"]), "y two-kernel")
    assert s.layer.get_error() == 0


def test_mxfp4_duplicates_and_bad_ids(dev):
    from sparse_expert_gemv_gb300 import MOE_DEVICE_BAD_ID
    # several tokens (two kernels)
    s = Small(dev, 6, 4, 256, 64, 4, fmt="mxfp4")
    ids = s.ids.copy()
    ids[0, 1] = ids[0, 0]
    ids[2, :] = ids[2, 0]
    ids[1, 3] = 6
    ids[3, 0] = -2
    h, _ = s.check(ids=ids)
    hb = tensor_to_f64(h)
    assert np.all(hb[1, 3] == 0) and np.all(hb[3, 0] == 0)
    assert s.layer.get_error() == MOE_DEVICE_BAD_ID
    # one token (one launch)
    s = Small(dev, 16, 4, 1024, 256, 1, seed=3, fmt="mxfp4")
    assert s.layer.fused_single_token
    ids = s.ids.copy()
    ids[0, 1] = ids[0, 0]
    ids[0, 3] = 99
    h, y = _layer_once(s, ids=ids)
    r = s.ref(ids=ids)
    assert np.all(tensor_to_f64(h)[0, 3] == 0)
    assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y")
    assert s.layer.get_error() == MOE_DEVICE_BAD_ID


def test_mxfp4_all_codes_one_hot(dev):
    # one expert whose gate/up codes run through all 16 E2M1 codes in every
    # block (both nibbles of every byte vary), scales 2^-17 .. 2^7; x is the
    # identity on one column per call, so each h is SiLU(g) * u of single
    # products and the GPU's h must match the oracle's
    E, k, H, I = 2, 1, 256, 32
    w = wl.Workload(91, "codes", E, k, H, I, 1, 0.05)
    rng = np.random.default_rng(5)
    experts = {}
    for e in range(E):
        wgu = rng.integers(0, 256, size=(2 * I, H // 2), dtype=np.uint8)
        sgu = rng.integers(110, 135, size=(2 * I, H // 32), dtype=np.uint8)
        wd = rng.integers(0, 256, size=(H, I // 2), dtype=np.uint8)
        sd = rng.integers(110, 135, size=(H, I // 32), dtype=np.uint8)
        experts[e] = (wgu, sgu, wd, sd)
    from sparse_expert_gemv_gb300 import MoEDecode
    layer = MoEDecode(*device_weights(w, experts, dev, fmt="mxfp4"), k=k, max_T=4, fmt="mxfp4")
    ids = np.array([[0], [1], [0], [1]], dtype=np.int32)
    tw = np.ones((4, 1), dtype=np.float32)
    for cols in ([0, 1, 2, 3], [30, 31, 32, 33], [126, 127, 254, 255]):
        xb = np.zeros((4, H), dtype=np.float32)
        for t, c in enumerate(cols):
            xb[t, c] = 1.0
        bits = torch.from_numpy(xb).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        x = bf16_tensor(bits, dev)
        h = layer.gate_up(x, torch.from_numpy(ids).to(dev))
        y = layer.down(h, torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev))
        torch.cuda.synchronize()
        r = oracle.layer(wl.bf16_bits_to_f64(bits), ids, tw, experts, E, H, I, fmt="mxfp4")
        assert_within(tensor_to_f64(h), r["h_spec"], 2.0 ** -7 * np.abs(r["h_spec"]) + 1e-30, "h")
        assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y")
    layer.close()


def test_mxfp4_host_path_and_noalloc(dev):
    from sparse_expert_gemv_gb300 import MOE_FLAG_HOST_COPY, MOE_FLAG_MXFP4, lib
    from sparse_expert_gemv_gb300._lib import MoEConfig
    a = Small(dev, 8, 4, 1024, 128, 1, fmt="mxfp4")
    c = Small(dev, 8, 4, 1024, 128, 1, fmt="mxfp4", flags=MOE_FLAG_HOST_COPY)
    assert a.layer.fused_single_token
    _, y_dev = _layer_once(a)
    want = y_dev.cpu().view(torch.int16)
    x = torch.from_numpy(a.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    ids = torch.from_numpy(a.ids).pin_memory()
    tw = torch.from_numpy(a.tw).pin_memory()
    assert torch.equal(a.layer.forward_host(x, ids, tw).view(torch.int16), want)
    assert torch.equal(c.layer.forward_host(x, ids, tw).view(torch.int16), want)
    # the allocation-free call with the MXFP4 flag, one token and several
    w = a.w
    cfg = MoEConfig(w.E, w.k, w.H, w.I, 0, MOE_FLAG_MXFP4)
    stream = torch.cuda.current_stream()
    for T, seed in ((1, 7), (5, 2)):
        xb = wl.make_x(w, seed, T)
        ids_np, tw_np = oracle.route(wl.make_logits(w, seed, T), w.k)
        xd = bf16_tensor(xb, dev)
        di = torch.from_numpy(ids_np).to(dev)
        dw = torch.from_numpy(tw_np).to(dev)
        y = torch.full((T, w.H), float("nan"), dtype=torch.bfloat16, device=dev)
        p = ctypes.c_void_p
        st = lib.moe_decode_layer_noalloc(ctypes.byref(cfg), *[p(t.data_ptr()) for t in a.wts], T,
                                          p(xd.data_ptr()), p(di.data_ptr()), p(dw.data_ptr()),
                                          p(y.data_ptr()), p(stream.cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        r = oracle.layer(wl.bf16_bits_to_f64(xb), ids_np, tw_np, a.experts, w.E, w.H, w.I,
                         fmt="mxfp4")
        assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), f"noalloc T={T}")


def test_mxfp4_shape_checks(dev):
    from sparse_expert_gemv_gb300 import MoEDecode
    w = wl.Workload(92, "shape", 4, 2, 256, 64, 1, 0.05)
    ex = wl.make_experts(w, 1, range(4), fmt="mxfp4")
    wts = device_weights(w, ex, dev, fmt="mxfp4")
    with pytest.raises(ValueError):
        MoEDecode(*wts, k=2, fmt="mxfp8")          # packed codes read as MXFP8: shapes disagree
    with pytest.raises(ValueError):
        MoEDecode(*wts, k=2, fmt="fp6")
