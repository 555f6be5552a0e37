"""The small-batch MoE decode layer, written out plainly in float64.

Source: the warp-decode post (cursor.com/blog/warp-decode).

  "The classic MoE path": every token is routed to k of E experts (e.g. 8 of
      128).
  "How the two kernels work": the gate/up kernel computes, for every
      (token, routed expert, intermediate neuron), the gate and up dot products
      of that neuron's two weight rows with the token's activation vector and
      writes one value SiLU(gate) * up. The down kernel computes, for every
      (token, output dimension), the routing-weighted sum over the token's
      top-k experts of that expert's down-projection row dotted with the
      intermediate activations.
  "Improved accuracy": activations stay BF16 and accumulators FP32.

Readings where the pages are silent:

  * W_gateup[e] is [2I, H]: rows [0, I) gate, rows [I, 2I) up.
  * SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)).
  * h[t, j, i] is stored as BF16 (round to nearest even); y[t, h] likewise.
  * The routing weight multiplies inside the down projection's sum, never h.
  * Routing: softmax over all E logits, the k largest probabilities (ties to
    the lower expert id, ids ordered by decreasing weight), renormalised to
    sum to one, stored as float32.
  * An expert id outside [0, E) contributes nothing: its h slice is zero and it
    adds nothing to y.
  * Duplicate ids in one token's row are legal and simply add up.

The oracle's float64 result is the exact layer up to float64 rounding; the
only precision it imitates is the BF16 storage of h ("h_spec"). "h_pure"/"y_pure"
skip that rounding and serve as the full-precision reference the accuracy
figures are measured against.
"""
from __future__ import annotations

from typing import Callable, Mapping

import numpy as np

from .bf16 import bf16_rne
from .mxfp4 import dequantize as dequantize_mxfp4
from .mxfp8 import E4M3, dequantize

ExpertSource = Mapping[int, tuple] | Callable[[int], tuple]


def _get(experts: ExpertSource, e: int):
    return experts(e) if callable(experts) else experts[e]


# Weight formats: MXFP8 (E4M3 codes, one byte each) and MXFP4 (E2M1 codes,
# two to a byte); both carry one UE8M0 scale per 32 elements along K.
def _float_weights(w, scales):
    """fmt "float": the expert holds full-precision weights (scales unused)."""
    return np.asarray(w, dtype=np.float64)


def _dq(fmt: str):
    if fmt == "mxfp8":
        return dequantize
    if fmt == "mxfp4":
        return dequantize_mxfp4
    if fmt == "float":
        return _float_weights
    raise ValueError(f"unknown weight format {fmt!r}")


def silu(z) -> np.ndarray:
    """z * sigmoid(z) in float64, evaluated without overflow for large |z|."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def route(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k routing: logits [T, E] -> (ids int32 [T, k], weights float32 [T, k]).

    Softmax over all E experts, keep the k most probable (ties to the lower id),
    renormalise the kept probabilities to sum to one.
    """
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-p[t, e], e))[:k]
        ids[t] = order
        kept = p[t, order]
        w[t] = (kept / kept.sum()).astype(np.float32)
    return ids, w


def dedup_schedule(ids: np.ndarray, E: int):
    """Per-step expert dedup: the unique routed experts and who uses each.

    Returns (uniq, off, pairs): uniq int32 [U] ascending expert ids; for the
    u-th unique expert, pairs[off[u]:off[u+1]] lists the flattened slots
    p = t*k + j (ascending) whose id equals uniq[u]. Out-of-range ids are
    left out.
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    users: dict[int, list[int]] = {}
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if 0 <= e < E:
                users.setdefault(e, []).append(t * k + j)
    uniq = sorted(users)
    off = [0]
    pairs: list[int] = []
    for e in uniq:
        pairs.extend(users[e])
        off.append(len(pairs))
    return (np.array(uniq, dtype=np.int32), np.array(off, dtype=np.int32),
            np.array(pairs, dtype=np.int32))


def _slots_by_expert(ids: np.ndarray, E: int, tokens) -> dict[int, list[tuple[int, int]]]:
    T, k = ids.shape
    by_e: dict[int, list[tuple[int, int]]] = {}
    for t in (range(T) if tokens is None else tokens):
        for j in range(k):
            e = int(ids[t, j])
            if 0 <= e < E:
                by_e.setdefault(e, []).append((t, j))
    return by_e


def gate_up(x: np.ndarray, ids: np.ndarray, experts: ExpertSource, E: int, I: int,
            tokens=None, fmt: str = "mxfp8") -> tuple[np.ndarray, np.ndarray]:
    """h[t, j, :] = SiLU(dq(Wg_e) x_t) * (dq(Wu_e) x_t), e = ids[t, j].

    x: float64 [T, H] holding the bf16 input values exactly.
    Returns (h_spec, h_pure), float64 [T, k, I]; h_spec is rounded to bf16.
    `tokens` restricts the work to a subset of tokens (other rows stay zero).
    Each expert is dequantised once and released after its slots are done.
    `fmt` names the weight format ("mxfp8" or "mxfp4").
    """
    dequantize = _dq(fmt)
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    T, k = ids.shape
    h_pure = np.zeros((T, k, I), dtype=np.float64)
    for e, slots in _slots_by_expert(ids, E, tokens).items():
        wgu, sgu = _get(experts, e)[:2]
        W = dequantize(wgu, sgu)
        for t, j in slots:
            gate = W[:I] @ x[t]
            up = W[I:] @ x[t]
            h_pure[t, j] = silu(gate) * up
        del W
    return bf16_rne(h_pure), h_pure


def down(h: np.ndarray, ids: np.ndarray, w: np.ndarray, experts: ExpertSource, E: int,
         H: int, tokens=None, rows=None, fmt: str = "mxfp8") -> np.ndarray:
    """y[t, r] = sum_j w[t, j] * (dq(Wd_e)[r, :] . h[t, j, :]), e = ids[t, j].

    h: float64 [T, k, I]; w: float32 [T, k] (used at its exact value).
    Returns float64 [T, H] (or [T, len(rows)]), not rounded.
    """
    dequantize = _dq(fmt)
    h = np.asarray(h, dtype=np.float64)
    ids = np.asarray(ids)
    wt = np.asarray(w, dtype=np.float32).astype(np.float64)
    T, k = ids.shape
    rows = np.arange(H) if rows is None else np.asarray(rows)
    terms = np.zeros((T, k, len(rows)), dtype=np.float64)
    for e, slots in _slots_by_expert(ids, E, tokens).items():
        wd, sd = _get(experts, e)[2:4]
        W = dequantize(wd[rows], None if sd is None else sd[rows])
        for t, j in slots:
            terms[t, j] = wt[t, j] * (W @ h[t, j])
        del W
    return terms.sum(axis=1)


def layer(x, ids, w, experts: ExpertSource, E: int, H: int, I: int, tokens=None, rows=None,
          fmt: str = "mxfp8"):
    """The whole layer: h_spec, h_pure, y_spec (from bf16 h), y_pure (from exact h)."""
    h_spec, h_pure = gate_up(x, ids, experts, E, I, tokens=tokens, fmt=fmt)
    y_spec = down(h_spec, ids, w, experts, E, H, tokens=tokens, rows=rows, fmt=fmt)
    y_pure = down(h_pure, ids, w, experts, E, H, tokens=tokens, rows=rows, fmt=fmt)
    return {"h_spec": h_spec, "h_pure": h_pure, "y_spec": y_spec, "y_pure": y_pure}


# ---------------------------------------------------------------------------
# The classic expert-centric path's extra rounding (warp-decode post,
# "Improved accuracy"): it converts the BF16 intermediate activations to MXFP8
# and back before the down projection. Used only to compare accuracies.
# ---------------------------------------------------------------------------

_FINITE = np.array([c for c in range(256) if np.isfinite(E4M3[c]) and E4M3[c] >= 0
                    and not (c == 0x80)], dtype=np.int64)
_POS_CODES = np.array(sorted(_FINITE, key=lambda c: E4M3[c]), dtype=np.int64)
_POS_VALS = E4M3[_POS_CODES]


def _round_e4m3(q: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value (ties to the even code), saturating at +-448."""
    q = np.asarray(q, dtype=np.float64)
    a = np.minimum(np.abs(q), 448.0)
    hi = np.searchsorted(_POS_VALS, a, side="left")
    hi = np.clip(hi, 0, len(_POS_VALS) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALS) - 1)
    vlo, vhi = _POS_VALS[lo], _POS_VALS[hi]
    dlo, dhi = a - vlo, vhi - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0))
    v = np.where(pick_hi, vhi, vlo)
    v = np.where(a == vhi, vhi, v)
    return np.copysign(v, q)


def requantize_mxfp8(a: np.ndarray) -> np.ndarray:
    """BF16 -> MXFP8 -> float64 along the last axis (blocks of 32).

    Shared exponent per block = floor(log2(amax)) - 8 clamped to [-127, 127];
    elements are divided by 2^exp, rounded to the nearest E4M3 value and scaled
    back.
    """
    a = np.asarray(a, dtype=np.float64)
    K = a.shape[-1]
    b = a.reshape(*a.shape[:-1], K // 32, 32)
    amax = np.abs(b).max(axis=-1)
    _, ex = np.frexp(amax)
    e = np.clip(ex - 1 - 8, -127, 127)
    e = np.where(amax == 0, 0, e)
    q = np.ldexp(b, -e[..., None])
    return np.ldexp(_round_e4m3(q), e[..., None]).reshape(a.shape)


def layer_classic(x, ids, w, experts: ExpertSource, E: int, H: int, I: int, tokens=None,
                  fmt: str = "mxfp8"):
    """Layer output when h is quantised to MXFP8 before the down projection."""
    h_spec, _ = gate_up(x, ids, experts, E, I, tokens=tokens, fmt=fmt)
    return down(requantize_mxfp8(h_spec), ids, w, experts, E, H, tokens=tokens, fmt=fmt)
