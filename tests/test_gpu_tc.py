"""GPU parity of the expert-centric tensor-core path (moe_tc_prep,
moe_tc_gate_up, moe_tc_down, moe_tc_combine: MX weights decoded exactly to
bf16 in tensor memory, tcgen05.mma kind::f16 with FP32 accumulators) against
the float64 oracle, with the tolerances of test_gpu_parity (one bf16 step of
h and y plus 1e-3 rms; y against the oracle's down projection of the
layer's own bf16 h, see TcCase.check):

  * a small layer (E=16, k=4, H=1024, I=256) with every output checked, at
    token counts giving one token, ragged column chunks, experts with more
    than 64 pairs (several chunks) and two token groups (T > 256), in both
    weight formats;
  * the batch shapes of the crossover study (E=128, k=8, H=2048, I=768 at
    T = 32, 64, 128, 256) on sampled tokens, the other tokens' experts holding
    finite marker weights;
  * duplicate and invalid ids, determinism, and when the path is available.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_within, bf16_tensor, device_weights, metrics, tensor_to_f64, tol_h, tol_y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


class TcCase:
    """A seeded layer whose checked tokens' experts hold seeded weights (all
    experts when every token is checked) and every other expert finite
    marker weights (device_weights fill="finite")."""

    def __init__(self, dev, E, k, H, I, T, seed, fmt="mxfp8", check=None, ids=None, sigma=0.02):
        from sparse_expert_gemv_gb300 import MoEDecode
        self.w = wl.Workload(91, "tensor-core case", E, k, H, I, T, sigma)
        self.T, self.fmt, self.dev = T, fmt, dev
        self.x_bits = wl.make_x(self.w, seed, T)
        rids, self.tw = oracle.route(wl.make_logits(self.w, seed, T), k)
        self.ids = rids if ids is None else np.ascontiguousarray(ids, dtype=np.int32)
        self.tokens = list(range(T)) if check is None else list(check)
        need = np.unique(self.ids[self.tokens])
        need = need[(need >= 0) & (need < E)]
        self.experts = wl.make_experts(self.w, seed, need, fmt=fmt)
        self.layer = MoEDecode(*device_weights(self.w, self.experts, dev, fmt=fmt, fill="finite"),
                               k=k, max_T=T, fmt=fmt)

    def run(self, path="tensor"):
        w = self.w
        self.layer.set_path(path)
        x = bf16_tensor(self.x_bits, self.dev)
        ids = torch.from_numpy(self.ids).to(self.dev)
        tw = torch.from_numpy(np.ascontiguousarray(self.tw, dtype=np.float32)).to(self.dev)
        h = torch.full((self.T, w.k, w.I), float("nan"), dtype=torch.bfloat16, device=self.dev)
        y = self.layer.layer(x, ids, tw, h=h)
        torch.cuda.synchronize()
        return h, y

    def check(self, h, y):
        """h against the oracle's h (one bf16 step), and y against the
        oracle's down projection of this h: the layer's y is defined from its
        stored bf16 intermediate h (the warp-decode post, "How the two kernels
        work"), and the tensor cores' FP32 sums, truncated after every 16
        products, put a few more h values on the other side of a bf16 rounding
        boundary than FP32 FMA chains do; each such h moves every y of its
        token, so y is compared with the y that this h defines."""
        w, S = self.w, self.tokens
        ref = oracle.layer(wl.bf16_bits_to_f64(self.x_bits), self.ids, self.tw, self.experts,
                           w.E, w.H, w.I, tokens=S, fmt=self.fmt)
        hg = tensor_to_f64(h)
        hm = assert_within(hg[S], ref["h_spec"][S], tol_h(ref["h_spec"][S]), "h")
        y_own = oracle.down(hg, self.ids, self.tw, self.experts, w.E, w.H, tokens=S, fmt=self.fmt)
        ym = assert_within(tensor_to_f64(y)[S], y_own[S], tol_y(y_own[S]), "y")
        return hm, ym, metrics(tensor_to_f64(y)[S], ref["y_pure"][S])


SMALL = (16, 4, 1024, 256)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("T", [1, 7, 64, 200, 300])
def test_small_layer_every_output(T, fmt, dev):
    # T=200: 800 pairs over 16 experts, about 50 each (ragged chunks, some
    # above 64); T=300: two token groups (256 + 44)
    c = TcCase(dev, *SMALL, T, seed=11 + T, fmt=fmt)
    assert c.layer.tensor_path
    h, y = c.run()
    assert c.layer.path(T) == "tensor"
    assert c.layer.kernel_name(T, "gate_up") == "moe_tc_gate_up"
    hm, ym, pure = c.check(h, y)
    print(f"{fmt} T={T}: h {hm}  y {ym}  y vs fp64-exact {pure}")
    assert pure["cosine"] > 0.9999
    assert c.layer.get_error() == 0


@pytest.mark.parametrize("T", [32, 64, 128, 256])
def test_crossover_shapes_sampled_tokens(T, dev):
    # the crossover study's layer shape; three tokens checked in full
    c = TcCase(dev, 128, 8, 2048, 768, T, seed=1002, check=[0, T // 2, T - 1])
    # the automatic choice: 1.5 or more routed slots per expert on average
    assert c.layer.path(T) == ("tensor" if 2 * T * 8 >= 3 * 128 else "warp")
    h, y = c.run()
    hm, ym, pure = c.check(h, y)
    print(f"T={T}: h {hm}  y {ym}  y vs fp64-exact {pure}")
    assert ym["cosine"] > 0.9999
    assert c.layer.get_error() == 0


def test_same_result_twice_and_from_auto(dev):
    c = TcCase(dev, *SMALL, 100, seed=5)
    h1, y1 = c.run("tensor")
    h2, y2 = c.run("auto")               # T = 100 >= 64: the same kernels
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    h3, y3 = c.run("warp")               # the other path: within tolerance of the oracle too
    c.check(h3, y3)


@pytest.mark.parametrize("fmt,sigma", [("mxfp8", 1e-7), ("mxfp8", 3e5), ("mxfp4", 1e-7),
                                       ("mxfp4", 1.5e4)])
def test_scales_outside_the_f16_range(sigma, fmt, dev):
    # weights whose gate/up scale codes fall outside the range in which every
    # weight is exact in f16 (113 .. 134 for MXFP8, 113 .. 140 for MXFP4) but
    # inside the bf16 one (tiny: codes near 100; huge: 139 and 141): the
    # gate/up kernel decodes them to bf16 instead, and the layer still
    # matches the oracle
    c = TcCase(dev, *SMALL, 64, seed=7, fmt=fmt, sigma=sigma)
    assert c.layer.tensor_path
    c.check(*c.run())


def test_one_hot_expert_gets_every_token(dev):
    # every token routes slot 0 to expert 3: 200 pairs of one expert, four
    # column chunks (64 + 64 + 64 + 8)
    T, (E, k, H, I) = 200, SMALL
    rng = np.random.default_rng(3)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    for t in range(T):
        row = [e for e in ids[t] if e != 3][:k - 1]
        ids[t] = [3] + row
    c = TcCase(dev, E, k, H, I, T, seed=21, ids=ids)
    c.check(*c.run())


def test_duplicate_and_invalid_ids(dev):
    T, (E, k, H, I) = 70, SMALL
    c0 = TcCase(dev, E, k, H, I, T, seed=31)
    ids = c0.ids.copy()
    ids[0, 1] = ids[0, 0]            # one expert twice for a token
    ids[5, :] = ids[5, 0]            # one expert in every slot
    ids[9, 2] = E                    # out of range
    ids[12, 0] = -1
    c = TcCase(dev, E, k, H, I, T, seed=31, ids=ids)
    h, y = c.run()
    c.check(h, y)
    hb = tensor_to_f64(h)
    assert np.all(hb[9, 2] == 0) and np.all(hb[12, 0] == 0)
    from sparse_expert_gemv_gb300 import MOE_DEVICE_BAD_ID
    assert c.layer.get_error() == MOE_DEVICE_BAD_ID


def test_every_id_invalid_gives_zero(dev):
    T, (E, k, H, I) = 9, SMALL
    c = TcCase(dev, E, k, H, I, T, seed=41, ids=np.full((T, k), E + 5, dtype=np.int32))
    h, y = c.run()
    assert torch.count_nonzero(y) == 0 and torch.count_nonzero(h) == 0
    c.layer.get_error()


def test_not_available_with_nan_codes_or_small_shapes(dev):
    from sparse_expert_gemv_gb300 import MoEDecode, MoEError
    w = wl.Workload(92, "nan fill", 8, 2, 1024, 256, 4, 0.02)
    ex = wl.make_experts(w, 3, [0, 1])
    lay = MoEDecode(*device_weights(w, ex, dev), k=2, max_T=4)   # NaN codes in the other experts
    assert not lay.tensor_path
    assert lay.path(100) == "warp"
    with pytest.raises(MoEError):
        lay.set_path("tensor")
    w2 = wl.Workload(93, "small H", 8, 2, 256, 128, 4, 0.02)     # H not a multiple of 512
    lay2 = MoEDecode(*device_weights(w2, wl.make_experts(w2, 3, range(8)), dev), k=2, max_T=4)
    assert not lay2.tensor_path
