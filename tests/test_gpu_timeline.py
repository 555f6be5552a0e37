"""The one-launch single-token layer's per-CTA timeline (the library built with
-DMOE_TIMELINE, libmoe_decode_timeline.so): each CTA stamps the GPU's global
nanosecond timer at its phases (moe_decode_timeline.h). These tests check the
stamps against the orders the kernel's waits impose (a stamp taken before an
action that another stamp's wait observes comes first), that the launch's
output still matches the oracle, and print the median phase times, the
breakdown every change to that kernel is judged against."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_within, bf16_tensor, device_weights, tensor_to_f64, tol_h, tol_y

pytestmark = pytest.mark.gpu

ENTRY, INPUTS, ROUTED, FIRST_ISSUE, FIRST_LANDED, GATE_UP_DONE, ARRIVING = range(7)
DOWN_LANDED, BARRIER, H_STAGED, DOWN_DONE, ISSUE_DONE = range(7, 12)
NAMES = ["entry", "inputs", "routed", "first_issue", "first_landed", "gate_up_done", "arriving",
         "down_landed", "barrier", "h_staged", "down_done", "issue_done"]
NSTAMPS = 16


@pytest.fixture(scope="module")
def tl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    b = __graft_entry__._build_module()
    if b.stale(b.OUT_TIMELINE):
        b.build(timeline=True)
    lib = ctypes.CDLL(b.OUT_TIMELINE)
    from sparse_expert_gemv_gb300._lib import MoEConfig
    p = ctypes.c_void_p
    lib.moe_decode_create.argtypes = [ctypes.POINTER(MoEConfig), p, p, p, p, ctypes.POINTER(p)]
    lib.moe_decode_destroy.argtypes = [p]
    lib.moe_decode_layer_timeline.argtypes = [p, p, p, p, p, p, p, p]
    lib.moe_decode_timeline_ctas.argtypes = [p]
    lib.moe_decode_fused_layer.argtypes = [p]
    lib.moe_decode_get_error.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
    return lib


def _run(tl, E, k, H, I, seed, reps=3):
    from sparse_expert_gemv_gb300._lib import MoEConfig
    dev = torch.device("cuda:0")
    w = wl.Workload(97, "timeline", E, k, H, I, 1, 0.02)
    x_bits = wl.make_x(w, seed)
    ids, tw = oracle.route(wl.make_logits(w, seed), k)
    experts = wl.make_experts(w, seed, np.unique(ids))
    wts = device_weights(w, experts, dev)
    h_ = ctypes.c_void_p()
    cfg = MoEConfig(E, k, H, I, 1, 0)
    assert tl.moe_decode_create(ctypes.byref(cfg), *[t.data_ptr() for t in wts], ctypes.byref(h_)) == 0
    try:
        assert tl.moe_decode_fused_layer(h_) == 1
        G = tl.moe_decode_timeline_ctas(h_)
        stamps = torch.zeros((G, NSTAMPS), dtype=torch.int64, device=dev)
        x = bf16_tensor(x_bits, dev)
        di = torch.from_numpy(ids).to(dev)
        dw = torch.from_numpy(tw).to(dev)
        h = torch.full((1, k, I), float("nan"), dtype=torch.bfloat16, device=dev)
        y = torch.full((1, H), float("nan"), dtype=torch.bfloat16, device=dev)
        s = torch.cuda.current_stream().cuda_stream
        for _ in range(reps):
            stamps.zero_()
            assert tl.moe_decode_layer_timeline(h_, x.data_ptr(), di.data_ptr(), dw.data_ptr(),
                                                h.data_ptr(), y.data_ptr(), stamps.data_ptr(), s) == 0
        torch.cuda.synchronize()
        flags = ctypes.c_uint32(0)
        assert tl.moe_decode_get_error(h_, ctypes.byref(flags)) == 0 and flags.value == 0
    finally:
        tl.moe_decode_destroy(h_)
    r = oracle.layer(wl.bf16_bits_to_f64(x_bits), ids, tw, experts, E, H, I)
    assert_within(tensor_to_f64(h), r["h_spec"], tol_h(r["h_spec"]), "h")
    assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y")
    return stamps.cpu().numpy()


def _check_order(st):
    G = st.shape[0]
    # at these shapes every CTA has gate/up neurons and down rows, so it
    # reaches every stamp
    for i in range(len(NAMES)):
        assert np.all(st[:, i] > 0), NAMES[i]
    # one thread's program order, or a wait that observes the earlier stamp's
    # action (the first tile lands after it is issued)
    for a, b in [(ENTRY, INPUTS), (INPUTS, ROUTED), (ROUTED, FIRST_ISSUE),
                 (FIRST_ISSUE, FIRST_LANDED), (FIRST_LANDED, GATE_UP_DONE),
                 (GATE_UP_DONE, ARRIVING), (ARRIVING, DOWN_LANDED), (DOWN_LANDED, BARRIER),
                 (BARRIER, H_STAGED), (H_STAGED, DOWN_DONE), (FIRST_ISSUE, ISSUE_DONE)]:
        bad = np.nonzero(st[:, a] > st[:, b])[0]
        assert bad.size == 0, f"{NAMES[a]} after {NAMES[b]} on CTAs {bad[:8]}"
    # the grid barrier is passed only after every CTA posted its arrival
    assert st[:, ARRIVING].max() <= st[:, BARRIER].min()
    span = st[:, DOWN_DONE].max() - st[:, ENTRY].min()
    assert 0 < span < 10_000_000, span
    return G


def _summary(st):
    t0 = st[:, ENTRY].min()
    rel = (st[:, :len(NAMES)] - t0) / 1e3
    return {NAMES[i]: round(float(np.median(rel[:, i])), 2) for i in range(len(NAMES))} | {
        "down_done_max": round(float(rel[:, DOWN_DONE].max()), 2)}


@pytest.mark.parametrize("E,k,H,I", [(64, 8, 2048, 768), (16, 4, 1024, 256)])
def test_timeline_stamps_are_ordered(tl, E, k, H, I):
    st = _run(tl, E, k, H, I, seed=E + k)
    G = _check_order(st)
    print(f"timeline E{E} k{k} H{H} I{I} ({G} CTAs), median us from the first entry:",
          _summary(st))
