"""GPU edge cases: empty and ragged shapes, duplicates, invalid ids, extreme
scales, one-hot inputs, invariants, determinism, graphs and the host path."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import (assert_within, bf16_tensor, device_weights, tensor_to_f64, tol_h, tol_y)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


class Small:
    """A small synthetic layer with every expert generated."""

    def __init__(self, dev, E, k, H, I, T, seed=7, sigma=0.05, flags=0, fmt="mxfp8"):
        from sparse_expert_gemv_gb300 import MoEDecode
        self.w = wl.Workload(90, "edge", E, k, H, I, T, sigma)
        self.seed = seed
        self.fmt = fmt
        self.experts = wl.make_experts(self.w, seed, range(E), fmt=fmt)
        self.wts = device_weights(self.w, self.experts, dev, fmt=fmt)
        self.layer = MoEDecode(*self.wts, k=k, max_T=max(T, 1), flags=flags, fmt=fmt)
        self.dev = dev
        self.x_bits = wl.make_x(self.w, seed, T)
        self.ids, self.tw = oracle.route(wl.make_logits(self.w, seed, T), k)

    def run(self, x_bits=None, ids=None, tw=None):
        x_bits = self.x_bits if x_bits is None else x_bits
        ids = self.ids if ids is None else ids
        tw = self.tw if tw is None else tw
        x = bf16_tensor(x_bits, self.dev)
        di = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(self.dev)
        dw = torch.from_numpy(np.ascontiguousarray(tw, dtype=np.float32)).to(self.dev)
        h = self.layer.gate_up(x, di)
        y = self.layer.down(h, di, dw)
        torch.cuda.synchronize()
        return h, y

    def ref(self, x_bits=None, ids=None, tw=None):
        x_bits = self.x_bits if x_bits is None else x_bits
        ids = self.ids if ids is None else ids
        tw = self.tw if tw is None else tw
        w = self.w
        return oracle.layer(wl.bf16_bits_to_f64(x_bits), ids, tw, self.experts, w.E, w.H, w.I,
                            fmt=self.fmt)

    def check(self, **kw):
        h, y = self.run(**kw)
        r = self.ref(**kw)
        assert_within(tensor_to_f64(h), r["h_spec"], tol_h(r["h_spec"]), "h")
        assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y")
        return h, y


@pytest.mark.parametrize("E,k,H,I,T", [
    (5, 3, 1184, 96, 5),      # H/32 = 37 blocks: ragged lanes; I/32 = 3; k odd; T < NT
    (16, 16, 64, 64, 3),      # k > 8 (wide slot masks)
    (8, 2, 256, 128, 37),     # T > 32: two token groups
    (3, 1, 32, 32, 1),        # smallest shapes
    (64, 8, 2048, 32, 6),     # I = 32: one block per row
    (4, 4, 96, 160, 33),      # every expert shared by many tokens, 2 groups
])
def test_ragged_shapes(dev, E, k, H, I, T):
    Small(dev, E, k, H, I, T).check()


def test_T_zero_is_a_noop(dev):
    s = Small(dev, 8, 2, 256, 128, 1)
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device=dev)
    ids = torch.zeros((0, 2), dtype=torch.int32, device=dev)
    h = s.layer.gate_up(x, ids)
    y = s.layer.down(h, ids, torch.zeros((0, 2), dtype=torch.float32, device=dev))
    assert h.numel() == 0 and y.numel() == 0


def test_duplicate_ids_add_up(dev):
    s = Small(dev, 6, 4, 256, 64, 4)
    ids = s.ids.copy()
    ids[0, 1] = ids[0, 0]
    ids[2, :] = ids[2, 0]
    s.check(ids=ids)


def test_out_of_range_id_contributes_nothing(dev):
    s = Small(dev, 6, 3, 256, 64, 3)
    ids = s.ids.copy()
    ids[1, 2] = 6
    ids[2, 0] = -4
    h, y = s.check(ids=ids)
    hb = tensor_to_f64(h)
    assert np.all(hb[1, 2] == 0) and np.all(hb[2, 0] == 0)
    from sparse_expert_gemv_gb300 import MOE_DEVICE_BAD_ID
    assert s.layer.get_error() == MOE_DEVICE_BAD_ID
    assert s.layer.get_error() == 0      # reading clears it


def test_one_hot_x_selects_weight_columns(dev):
    s = Small(dev, 4, 2, 2048, 64, 4)
    for c in [0, 31, 32, 1023, 1024, 2047]:
        xb = np.zeros((4, 2048), dtype=np.float32)
        xb[:, c] = 1.0
        bits = torch.from_numpy(xb).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        h, _ = s.run(x_bits=bits)
        r = s.ref(x_bits=bits)
        # each dot has one product (exact in FP32): only SiLU's FP32 rounding differs
        assert_within(tensor_to_f64(h), r["h_spec"], 2.0 ** -7 * np.abs(r["h_spec"]) + 1e-30, "h")


def test_extreme_scales_bitwise_through_down(dev):
    # one expert whose down rows r carry (code, scale) pairs at block 1 and a
    # one-hot h selecting column 40 (block 1, element 8): y[r] = bf16(E4M3 * 2^(s-127)),
    # a single product, exact in FP32 unless it overflows (then inf on both sides)
    from sparse_expert_gemv_gb300 import MoEDecode
    E, k, H, I = 1, 1, 64, 64
    pairs = [(0x01, 0), (0x7E, 0), (0x38, 0), (0x08, 1), (0x7E, 254), (0x38, 254), (0xB8, 200),
             (0x01, 100), (0x00, 254), (0x07, 5), (0xFE, 130), (0x3C, 127)]
    wd = np.zeros((H, I), np.uint8)
    sd = np.full((H, I // 32), 127, np.uint8)
    for r, (c, s) in enumerate(pairs):
        wd[r, 40] = c
        sd[r, 1] = s
    experts = {0: (np.zeros((2 * I, H), np.uint8), np.full((2 * I, H // 32), 127, np.uint8), wd, sd)}
    wts = device_weights(wl.Workload(91, "x", E, k, H, I, 1, 0.0), experts, dev)
    layer = MoEDecode(*wts, k=1, max_T=1)
    h = torch.zeros((1, 1, I), dtype=torch.bfloat16, device=dev)
    h[0, 0, 40] = 1.0
    y = layer.down(h, torch.zeros((1, 1), dtype=torch.int32, device=dev),
                   torch.ones((1, 1), dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    got = tensor_to_f64(y)[0]
    want = oracle.bf16_rne(oracle.dequantize(wd, sd)[:, 40])
    assert np.array_equal(got[:len(pairs)], want[:len(pairs)]), (got[:len(pairs)], want[:len(pairs)])


def test_zero_routing_weight_and_topk_order(dev):
    s = Small(dev, 8, 4, 512, 96, 5)
    tw = s.tw.copy()
    tw[:, 2] = 0
    s.check(tw=tw)
    perm = [3, 1, 0, 2]
    _, y1 = s.run()
    _, y2 = s.run(ids=s.ids[:, perm], tw=s.tw[:, perm])
    ref = s.ref()["y_spec"]
    assert_within(tensor_to_f64(y2), tensor_to_f64(y1), tol_y(ref), "y permuted top-k")


def test_bitwise_deterministic_and_graph_capture(dev):
    s = Small(dev, 16, 4, 1024, 256, 8)
    h1, y1 = s.run()
    h2, y2 = s.run()
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    x = bf16_tensor(s.x_bits, dev)
    ids = torch.from_numpy(s.ids).to(dev)
    tw = torch.from_numpy(s.tw).to(dev)
    h = torch.empty_like(h1)
    y = torch.empty_like(y1)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        s.layer.layer(x, ids, tw, h=h, y=y)       # warm up outside capture
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    y.zero_()
    with torch.cuda.graph(g):
        s.layer.layer(x, ids, tw, h=h, y=y)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y1.view(torch.int16))


def test_no_pdl_flag_and_host_path(dev):
    from sparse_expert_gemv_gb300 import MOE_FLAG_HOST_COPY, MOE_FLAG_NO_PDL
    a = Small(dev, 8, 4, 512, 128, 6)
    b = Small(dev, 8, 4, 512, 128, 6, flags=MOE_FLAG_NO_PDL)
    c = Small(dev, 8, 4, 512, 128, 6, flags=MOE_FLAG_HOST_COPY)
    _, ya = a.run()
    _, yb = b.run()
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
    want = ya.cpu().view(torch.int16)
    x = torch.from_numpy(a.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    ids = torch.from_numpy(a.ids).pin_memory()
    tw = torch.from_numpy(a.tw).pin_memory()
    # pinned host buffers, read and written in place by the kernels
    yh = a.layer.forward_host(x, ids, tw)
    assert torch.equal(yh.view(torch.int16), want)
    # pageable host buffers: in place where the device reaches pageable
    # memory, else through the staging copies; same result
    yp = torch.empty_like(yh, pin_memory=False)
    a.layer.forward_host(x.clone(), ids.clone(), tw.clone(), y=yp)
    assert not yp.is_pinned()
    assert torch.equal(yp.view(torch.int16), want)
    # the staging copies, forced
    for xx, ii, ww in ((x, ids, tw), (x.clone(), ids.clone(), tw.clone())):
        yc = c.layer.forward_host(xx, ii, ww)
        assert torch.equal(yc.view(torch.int16), want)


def test_get_error_waits_for_its_own_work_only(dev):
    # a long kernel on another stream keeps running while the handle's error
    # word is read: the read waits for the handle's latest call (or a given
    # stream), not for the whole device
    import time
    from sparse_expert_gemv_gb300 import MOE_DEVICE_BAD_ID
    s = Small(dev, 8, 2, 256, 128, 1, seed=5)      # two-kernel path (no cooperative launch)
    assert not s.layer.fused_single_token
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(3_000_000_000)            # ~1.5 s of SM clock cycles at 2 GHz
    ids = s.ids.copy()
    ids[0, 1] = 77                                  # out of range: latches a flag
    x = bf16_tensor(s.x_bits, dev)
    di = torch.from_numpy(ids).to(dev)
    dw = torch.from_numpy(s.tw).to(dev)
    t0 = time.perf_counter()
    s.layer.layer(x, di, dw)
    flags = s.layer.get_error()
    dt = time.perf_counter() - t0
    busy = not side.query()
    assert flags == MOE_DEVICE_BAD_ID
    assert busy, "the side kernel finished before the error was read; cannot tell"
    assert dt < 0.5, f"get_error took {dt:.3f} s: it waited for another stream"
    # the stream-scoped form waits for the given stream
    s.layer.layer(x, di, dw)
    assert s.layer.get_error(stream=torch.cuda.current_stream()) == MOE_DEVICE_BAD_ID
    assert not side.query()
    side.synchronize()
    assert s.layer.get_error() == 0


def test_bad_arguments_raise(dev):
    from sparse_expert_gemv_gb300 import MoEError
    s = Small(dev, 8, 2, 256, 128, 2)
    x = bf16_tensor(s.x_bits, dev)
    ids = torch.from_numpy(s.ids).to(dev)
    big = torch.zeros((3, 256), dtype=torch.bfloat16, device=dev)
    with pytest.raises(MoEError):
        s.layer.gate_up(big, torch.zeros((3, 2), dtype=torch.int32, device=dev))   # T > max_T
    mis = torch.zeros(2 * 256 + 8, dtype=torch.bfloat16, device=dev)[8:].view(2, 256)
    with pytest.raises(MoEError):
        s.layer.gate_up(mis, ids)                                                  # 16-byte offset


# ---------------------------------------------------------------------------
# single-token layer calls (one persistent launch for both projections)
# ---------------------------------------------------------------------------

def _layer_once(s, ids=None, tw=None, x_bits=None):
    x = bf16_tensor(s.x_bits if x_bits is None else x_bits, s.dev)
    di = torch.from_numpy(np.ascontiguousarray(s.ids if ids is None else ids, dtype=np.int32)).to(s.dev)
    dw = torch.from_numpy(np.ascontiguousarray(s.tw if tw is None else tw, dtype=np.float32)).to(s.dev)
    h = torch.full((1, s.w.k, s.w.I), float("nan"), dtype=torch.bfloat16, device=s.dev)
    y = s.layer.layer(x, di, dw, h=h)
    torch.cuda.synchronize()
    return h, y


@pytest.mark.parametrize("E,k,H,I", [(8, 2, 512, 128), (16, 4, 1024, 256), (64, 8, 2048, 768),
                                     (12, 8, 7168, 2048), (6, 5, 1536, 384)])
def test_single_token_layer_matches_oracle(dev, E, k, H, I):
    s = Small(dev, E, k, H, I, 1, seed=E + H)
    assert s.layer.fused_single_token, "one-token layer calls should run as one launch here"
    h, y = _layer_once(s)
    r = s.ref()
    assert_within(tensor_to_f64(h), r["h_spec"], tol_h(r["h_spec"]), "h")
    assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y")
    # the two-kernel path on the same inputs agrees within the same bound
    _, y2 = s.run()
    assert_within(tensor_to_f64(y2), r["y_spec"], tol_y(r["y_spec"]), "y two-kernel")
    assert s.layer.get_error() == 0


def test_single_token_layer_duplicates_and_bad_ids(dev):
    from sparse_expert_gemv_gb300 import MOE_DEVICE_BAD_ID
    s = Small(dev, 16, 4, 1024, 256, 1, seed=3)
    assert s.layer.fused_single_token
    ids = s.ids.copy()
    ids[0, 1] = ids[0, 0]          # duplicate
    ids[0, 3] = 99                 # out of range
    h, y = _layer_once(s, ids=ids)
    r = s.ref(ids=ids)
    assert np.all(tensor_to_f64(h)[0, 3] == 0)
    assert_within(tensor_to_f64(h), r["h_spec"], tol_h(r["h_spec"]), "h")
    assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y")
    assert s.layer.get_error() == MOE_DEVICE_BAD_ID
    # every id out of range: y is all zeros
    h, y = _layer_once(s, ids=np.full((1, 4), -1, np.int32))
    assert torch.count_nonzero(y).item() == 0
    assert torch.count_nonzero(h).item() == 0
    assert s.layer.get_error() == MOE_DEVICE_BAD_ID
    # and the next call is fine again
    h, y = _layer_once(s)
    r = s.ref()
    assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y after")
    assert s.layer.get_error() == 0


def test_single_token_layer_graph_replays(dev):
    s = Small(dev, 64, 8, 2048, 768, 1, seed=11)
    assert s.layer.fused_single_token
    x = bf16_tensor(s.x_bits, dev)
    ids = torch.from_numpy(s.ids).to(dev)
    tw = torch.from_numpy(s.tw).to(dev)
    h = torch.empty((1, 8, 768), dtype=torch.bfloat16, device=dev)
    y = torch.empty((1, 2048), dtype=torch.bfloat16, device=dev)
    s.layer.layer(x, ids, tw, h=h, y=y)
    torch.cuda.synchronize()
    ref = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            s.layer.layer(x, ids, tw, h=h, y=y)
    for _ in range(4):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert s.layer.get_error() == 0


def test_single_token_layer_barrier_timeout_is_reported(dev):
    # failure detection without a fault: the grid barrier's bounded wait runs
    # out (the launch counter is moved out of its reach), every CTA gives up
    # after its bound, the launch completes and the handle reports
    # MOE_DEVICE_TIMEOUT; reading the error resets the counters and the next
    # call is correct again
    from sparse_expert_gemv_gb300 import MOE_DEVICE_TIMEOUT
    s = Small(dev, 16, 4, 1024, 256, 1, seed=21)
    assert s.layer.fused_single_token
    r = s.ref()
    _, y = _layer_once(s)
    assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y before")
    assert s.layer.get_error() == 0
    s.layer.arm_barrier_timeout()
    _layer_once(s)                                   # y unspecified
    assert s.layer.get_error() == MOE_DEVICE_TIMEOUT
    assert s.layer.get_error() == 0                  # reading clears it
    for _ in range(3):
        _, y = _layer_once(s)
        assert_within(tensor_to_f64(y), r["y_spec"], tol_y(r["y_spec"]), "y after")
    assert s.layer.get_error() == 0


# ---------------------------------------------------------------------------
# sixteen or more tokens with H a multiple of 512 (1024 for MXFP4): the
# gate/up projection streams 16-neuron tiles with TMA and forms the products
# on the warp-level MMA, items split over the CTAs (an expert's tokens in
# passes of eight)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("E,k,H,I,T", [
    (16, 4, 1024, 256, 20),   # a few tokens per expert
    (40, 12, 1024, 64, 24),   # k > 8, I = 64: four tiles per expert
    (6, 2, 1024, 32, 32),     # ~10 tokens per expert: two passes; I = 32
    (3, 3, 2048, 96, 17),     # every expert serves every token: three passes
])
def test_several_token_tma_gate_up(dev, fmt, E, k, H, I, T):
    from sparse_expert_gemv_gb300 import MOE_FLAG_WARP_MMA
    s = Small(dev, E, k, H, I, T, seed=E * T, fmt=fmt, flags=MOE_FLAG_WARP_MMA)
    s.layer.set_path("warp")        # layer calls too (the names are the layer call's kernels)
    assert s.layer.kernel_name(T, "gate_up") == "moe_gate_up_tma"
    s.check()
    ids = s.ids.copy()
    ids[0, 1 % k] = ids[0, 0]       # duplicate
    ids[T - 1, 0] = E + 2           # out of range
    ids[T // 2, k - 1] = -1
    h, _ = s.check(ids=ids)
    hb = tensor_to_f64(h)
    assert np.all(hb[T - 1, 0] == 0) and np.all(hb[T // 2, k - 1] == 0)
    from sparse_expert_gemv_gb300 import MOE_DEVICE_BAD_ID
    assert s.layer.get_error() == MOE_DEVICE_BAD_ID
    # bitwise reproducible
    h2, y2 = s.run(ids=ids)
    h3, y3 = s.run(ids=ids)
    assert torch.equal(h2.view(torch.int16), h3.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), y3.view(torch.int16))


# ---------------------------------------------------------------------------
# two or more tokens with I a multiple of 128 (at most 2048): the down
# projection streams each distinct routed expert's 16-row tiles with TMA,
# one warp per output row
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("E,k,H,I,T", [
    (8, 2, 256, 128, 2),      # the smallest tile counts
    (12, 10, 512, 384, 9),    # k > 8
    (20, 4, 96, 2048, 3),     # I at its maximum, six row tiles
    (6, 3, 256, 128, 40),     # T > 32: two token groups
])
@pytest.mark.parametrize("mma", [False, True])
def test_several_token_tma_down(dev, fmt, E, k, H, I, T, mma):
    from sparse_expert_gemv_gb300 import MOE_FLAG_WARP_MMA
    s = Small(dev, E, k, H, I, T, seed=3 * E + T, fmt=fmt, flags=MOE_FLAG_WARP_MMA if mma else 0)
    s.layer.set_path("warp")        # layer calls too (the names are the layer call's kernels)
    # token by token; with MOE_FLAG_WARP_MMA and 16 or more tokens (here a
    # group of 32) each unique expert's rows once, on the MMA
    assert s.layer.kernel_name(T, "down") == ("moe_down_mma" if mma and T >= 16 else "moe_down_tma")
    s.check()
    ids = s.ids.copy()
    ids[0, 1] = ids[0, 0]           # duplicate: one distinct expert, weights summed
    ids[T - 1, :] = ids[T - 1, 0]   # every slot the same expert
    ids[T // 2, k - 1] = E          # out of range
    _, y = s.check(ids=ids)
    from sparse_expert_gemv_gb300 import MOE_DEVICE_BAD_ID
    assert s.layer.get_error() == MOE_DEVICE_BAD_ID
    # every id of a token invalid: its y row is zero
    ids[1, :] = -1
    _, y = s.check(ids=ids)
    assert torch.count_nonzero(y[1]).item() == 0
    _, y2 = s.run(ids=ids)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_kernel_choice_by_workload(dev):
    # which kernels the seeded workloads' calls take (weights need not be real)
    from sparse_expert_gemv_gb300 import MoEDecode
    # (NaN weights: the tensor-core path is unavailable, so the warp path's
    # kernels are reported; the layer of workload 3 takes the tensor-core
    # path when the weights allow it, see test_gpu_tc.py)
    from sparse_expert_gemv_gb300 import MOE_FLAG_WARP_MMA
    want = {
        0: ("moe_gate_up_3d_batched", "moe_down_3d_batched"),       # T = 1, shapes below the ring kernels
        1: ("moe_gate_up_3d_batched", "moe_down_3d_batched"),       # T = 1 (moe_decode_layer: one launch)
        2: ("moe_gate_up_3d_batched_xs", "moe_down_tma"),
        3: ("moe_gate_up_3d_batched_xs", "moe_down_tma"),
    }
    for c, (gu, dn) in want.items():
        w = wl.workload(c)
        for fmt in ("mxfp8", "mxfp4"):
            lay = MoEDecode(*device_weights(w, {}, dev, fmt=fmt), k=w.k, max_T=w.T, fmt=fmt)
            assert lay.kernel_name(w.T, "gate_up") == gu, (c, fmt)
            assert lay.kernel_name(w.T, "down") == dn, (c, fmt)
            if c == 3:
                # the warp-level MMA kernels when asked for
                lay.close()
                lay = MoEDecode(*device_weights(w, {}, dev, fmt=fmt), k=w.k, max_T=w.T, fmt=fmt,
                                flags=MOE_FLAG_WARP_MMA)
                assert lay.kernel_name(w.T, "gate_up") == "moe_gate_up_tma", fmt
                assert lay.kernel_name(w.T, "down") == "moe_down_mma", fmt
            # the one-launch single-token form depends on the shape alone
            assert lay.fused_single_token == (c != 0), (c, fmt)
            lay.close()
