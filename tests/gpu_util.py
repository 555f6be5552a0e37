"""Helpers for the GPU parity tests: device copies of seeded layers, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def device_weights(w: wl.Workload, experts: dict, device, fill_code=wl.NAN_CODE, fmt="mxfp8",
                   fill="nan"):
    """Full [E, ...] device tensors; experts absent from `experts` hold NaN codes
    (MXFP8) or NaN scales (MXFP4, whose codes have no NaN), so a kernel that
    reads them poisons exactly the outputs that used them. With fill="finite"
    they hold the value 1.0 * 2^-7 everywhere instead (code 0x38 or the E2M1
    pair 0x22, scale 120): finite, so the tensor-core path stays available,
    yet far from the seeded weights, so reading them still shows in the
    outputs that used them."""
    E, H, I = w.E, w.H, w.I
    per = 2 if fmt == "mxfp4" else 1
    fill_scale = 127
    if fill == "finite":
        fill_code, fill_scale = (0x22 if fmt == "mxfp4" else 0x38), 120
    elif fmt == "mxfp4":
        fill_code, fill_scale = 0x77, 0xFF
    wgu = torch.full((E, 2 * I, H // per), fill_code, dtype=torch.uint8, device=device)
    sgu = torch.full((E, 2 * I, H // 32), fill_scale, dtype=torch.uint8, device=device)
    wd = torch.full((E, H, I // per), fill_code, dtype=torch.uint8, device=device)
    sd = torch.full((E, H, I // 32), fill_scale, dtype=torch.uint8, device=device)
    for e, (a, b, c, d) in experts.items():
        wgu[e].copy_(torch.from_numpy(a))
        sgu[e].copy_(torch.from_numpy(b))
        wd[e].copy_(torch.from_numpy(c))
        sd[e].copy_(torch.from_numpy(d))
    return wgu, sgu, wd, sd


def tol_y(ref: np.ndarray) -> np.ndarray:
    """|y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref)."""
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return 2.0 ** -7 * np.abs(ref) + 1e-3 * rms


def tol_h(ref: np.ndarray) -> np.ndarray:
    """|h - h_spec| <= 2^-7 |h_spec| + 1e-3 rms(h_spec).

    h is stored in bf16 (8 significant bits). When the GPU's FP32 value and the
    oracle's float64 value fall on opposite sides of a rounding midpoint, the
    two bf16 results are one step apart, and one step is at most 2^-7 of the
    value (at the bottom of a binade).
    """
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return 2.0 ** -7 * np.abs(ref) + 1e-3 * rms


def assert_within(got: np.ndarray, ref: np.ndarray, tol: np.ndarray, what: str) -> dict:
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside tolerance, "
                           f"worst {float(err.max()):.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return metrics(got, ref)


def metrics(got: np.ndarray, ref: np.ndarray) -> dict:
    g, r = got.ravel(), ref.ravel()
    nr = float(np.linalg.norm(r))
    cos = float(g @ r / (np.linalg.norm(g) * nr)) if nr > 0 else 1.0
    return {"rel_l2": float(np.linalg.norm(g - r) / nr) if nr > 0 else 0.0,
            "cosine": cos, "max_abs": float(np.abs(g - r).max()) if g.size else 0.0}


class Case:
    """A seeded workload with its routing and the experts it needs."""

    def __init__(self, c: int, T: int | None = None, tokens=None, fmt: str = "mxfp8"):
        self.fmt = fmt
        self.w = w = wl.workload(c)
        self.seed = wl.seed_of(c)
        self.T = w.T if T is None else T
        self.x_bits = wl.make_x(w, self.seed, self.T)
        self.logits = wl.make_logits(w, self.seed, self.T)
        self.ids, self.tw = oracle.route(self.logits, w.k)
        self.tokens = list(range(self.T)) if tokens is None else list(tokens)
        need = np.unique(self.ids[self.tokens])
        self.experts = wl.make_experts(w, self.seed, need, fmt=fmt)

    def x64(self):
        return wl.bf16_bits_to_f64(self.x_bits)

    def ref(self):
        w = self.w
        return oracle.layer(self.x64(), self.ids, self.tw, self.experts, w.E, w.H, w.I,
                            tokens=self.tokens, fmt=self.fmt)


def check_layer_call(layer, case, x, ids, tw, y_two, fmt="mxfp8") -> None:
    """The layer entry point on a case whose gate/up + down results (y_two)
    were already checked: at T = 1 through the one-launch kernel, y against
    the oracle; on the tensor-core path, h against the oracle's h and y
    against the oracle's down projection of that h (the layer's y is defined
    from its stored bf16 h, and the tensor cores' FP32 sums put a few more h
    values on the other side of a bf16 rounding boundary than FMA chains
    do); otherwise bit for bit the two-kernel result."""
    w, S = case.w, case.tokens
    h2 = torch.full((case.T, w.k, w.I), float("nan"), dtype=torch.bfloat16, device=x.device)
    y2 = layer.layer(x, ids, tw, h=h2)
    torch.cuda.synchronize()
    ref = case.ref()
    if case.T == 1 and layer.fused_single_token:
        # one launch for both projections: its own sums, checked on their own
        assert_within(tensor_to_f64(y2)[S], ref["y_spec"][S], tol_y(ref["y_spec"][S]),
                      "y (one launch)")
    elif layer.path(case.T) == "tensor":
        hg = tensor_to_f64(h2)
        assert_within(hg[S], ref["h_spec"][S], tol_h(ref["h_spec"][S]), "h (tensor cores)")
        y_own = oracle.down(hg, case.ids, case.tw, case.experts, w.E, w.H, tokens=S, fmt=fmt)
        assert_within(tensor_to_f64(y2)[S], y_own[S], tol_y(y_own[S]), "y (tensor cores)")
    else:
        assert torch.equal(y_two.view(torch.int16)[S], y2.view(torch.int16)[S]), \
            "layer() differs from gate_up+down"
