"""Pins for the oracle's layer arithmetic: routing, dedup schedule, gate/up, down.

Each pin is independent of the code it checks: brute-force scalar loops that
decode through torch's float8 types and sum with math.fsum, a dense special
case against numpy matmul, library routines (scipy softmax, torch SiLU) and
invariants of the layer. The mutation tests at the end plant plausible
mistakes in the oracle and check that a pin catches each one.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import oracle.moe as om
import workloads as wl

# ---------------------------------------------------------------------------
# independent decoders and a brute-force layer (scalar Python loops)
# ---------------------------------------------------------------------------

_EV = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).tolist()
_SV = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).tolist()


def _w(codes, scales, r, K):
    return _EV[int(codes[r, K])] * _SV[int(scales[r, K // 32])]


def _silu(z):
    if z >= 0:
        return z / (1.0 + math.exp(-z))
    ez = math.exp(z)
    return z * ez / (1.0 + ez)


def brute_layer(x, ids, w, experts, E, H, I):
    """Returns (h_pure, y_pure) from scalar loops with exact (fsum) dot products."""
    T, k = ids.shape
    h = np.zeros((T, k, I))
    y = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if not 0 <= e < E:
                continue
            wgu, sgu, wd, sd = experts[e]
            for i in range(I):
                g = math.fsum(_w(wgu, sgu, i, K) * x[t, K] for K in range(H))
                u = math.fsum(_w(wgu, sgu, I + i, K) * x[t, K] for K in range(H))
                h[t, j, i] = _silu(g) * u
        for r in range(H):
            terms = []
            for j in range(k):
                e = int(ids[t, j])
                if not 0 <= e < E:
                    continue
                wd, sd = experts[e][2], experts[e][3]
                terms.append(float(w[t, j]) * math.fsum(_w(wd, sd, r, K) * h[t, j, K] for K in range(I)))
            y[t, r] = math.fsum(terms)
    return h, y


def tiny_case(E, k, H, I, T, seed, sigma=0.05):
    w = wl.Workload(99, "tiny", E, k, H, I, T, sigma)
    x = wl.bf16_bits_to_f64(wl.make_x(w, seed))
    ids, wt = oracle.route(wl.make_logits(w, seed), k)
    experts = wl.make_experts(w, seed, range(E), threads=1)
    return w, x, ids, wt, experts


def close(a, b, rel=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    scale = max(np.abs(b).max(), 1e-300)
    return np.abs(a - b).max() <= rel * scale


# ---------------------------------------------------------------------------
# SiLU, routing, dedup
# ---------------------------------------------------------------------------

def test_silu_matches_torch():
    z = np.concatenate([np.linspace(-50, 50, 2001), [-800.0, -1e-300, 0.0, 1e-300, 800.0]])
    want = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    got = oracle.silu(z)
    assert np.allclose(got, want, rtol=1e-15, atol=1e-300)
    assert np.all(np.isfinite(got))


def test_route_against_topk_of_logits():
    # top-k of the softmax = top-k of the logits (exp is increasing), and the
    # renormalised weights equal a softmax over the k kept logits alone
    rng = np.random.default_rng(11)
    for E, k, T in [(8, 2, 5), (128, 8, 32), (256, 8, 3), (5, 5, 4)]:
        logits = rng.standard_normal((T, E)).astype(np.float32)
        ids, w = oracle.route(logits, k)
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
            assert list(ids[t]) == order
            kept = logits[t, order].astype(np.float64)
            sm = scipy.special.softmax(kept)
            assert np.allclose(w[t], sm, rtol=2e-7, atol=0)
            assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6


def test_route_full_softmax_matches_scipy():
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((4, 16)).astype(np.float32)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    ids, w = oracle.route(logits, 16)       # k = E keeps everything
    for t in range(4):
        assert np.allclose(w[t], p[t, ids[t]], rtol=2e-7)


def test_route_ties_go_to_lower_id():
    logits = np.zeros((1, 6), np.float32)
    logits[0, [1, 4]] = 1.0
    ids, w = oracle.route(logits, 4)
    assert list(ids[0]) == [1, 4, 0, 2]


def test_dedup_schedule_brute_force():
    rng = np.random.default_rng(13)
    for E, k, T in [(8, 2, 1), (128, 8, 32), (16, 8, 8), (4, 3, 7)]:
        ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        ids[0, 0] = -1 if T > 1 else ids[0, 0]      # one out-of-range id
        uniq, off, pairs = oracle.dedup_schedule(ids, E)
        flat = ids.reshape(-1)
        valid = (flat >= 0) & (flat < E)
        assert list(uniq) == sorted(np.unique(flat[valid]).tolist())
        assert off[0] == 0 and off[-1] == valid.sum()
        for u, e in enumerate(uniq):
            assert list(pairs[off[u]:off[u + 1]]) == np.flatnonzero(flat == e).tolist()


# ---------------------------------------------------------------------------
# layer: brute force, dense special case
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("E,k,H,I,T", [(1, 1, 32, 32, 1), (2, 2, 64, 32, 2), (4, 2, 32, 64, 3),
                                       (4, 1, 64, 64, 1)])
def test_layer_brute_force_tiny(E, k, H, I, T):
    w, x, ids, wt, experts = tiny_case(E, k, H, I, T, seed=50 + E + H)
    out = oracle.layer(x, ids, wt, experts, E, H, I)
    h_bf, y_bf = brute_layer(x, ids, wt, experts, E, H, I)
    assert close(out["h_pure"], h_bf)
    assert close(out["y_pure"], y_bf)
    # h_spec is h_pure rounded to bf16 (torch's own float32->bf16 rounding of
    # the float32-representable h values, where they are representable)
    assert np.array_equal(out["h_spec"], oracle.bf16_rne(out["h_pure"]))


def test_layer_brute_force_workload0():
    w = wl.workload(0)
    s = wl.seed_of(0)
    x = wl.bf16_bits_to_f64(wl.make_x(w, s))
    ids, wt = oracle.route(wl.make_logits(w, s), w.k)
    experts = wl.make_experts(w, s, np.unique(ids))
    out = oracle.layer(x, ids, wt, experts, w.E, w.H, w.I)
    h_bf, y_bf = brute_layer(x, ids, wt, experts, w.E, w.H, w.I)
    assert close(out["h_pure"], h_bf)
    assert close(out["y_pure"], y_bf)


def test_dense_special_case_matches_matmul():
    # E = 1, k = 1, w = 1: the layer is y = Wd (silu(Wg x) * (Wu x))
    H, I = 128, 64
    w = wl.Workload(98, "dense", 1, 1, H, I, 1, 0.03)
    wgu, sgu, wd, sd = wl.make_expert(w, 77, 0)

    def tdq(codes, scales):
        v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
        s = torch.from_numpy(scales).view(torch.float8_e8m0fnu).to(torch.float64)
        return (v * s.repeat_interleave(32, dim=1)).numpy()

    Wgu, Wd = tdq(wgu, sgu), tdq(wd, sd)
    x = wl.bf16_bits_to_f64(wl.make_x(w, 77))[0]
    hh = torch.nn.functional.silu(torch.from_numpy(Wgu[:I] @ x)).numpy() * (Wgu[I:] @ x)
    y = Wd @ hh
    out = oracle.layer(x[None], np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32),
                       {0: (wgu, sgu, wd, sd)}, 1, H, I)
    assert close(out["h_pure"][0, 0], hh, 1e-13)
    assert close(out["y_pure"][0], y, 1e-13)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def mid_case():
    return tiny_case(E=6, k=3, H=64, I=96, T=4, seed=123)


def test_zero_weight_removes_expert(mid_case):
    w, x, ids, wt, experts = mid_case
    h, _ = oracle.gate_up(x, ids, experts, w.E, w.I)
    y = oracle.down(h, ids, wt, experts, w.E, w.H)
    wt0 = wt.copy(); wt0[:, 1] = 0
    y0 = oracle.down(h, ids, wt0, experts, w.E, w.H)
    contrib = np.stack([float(wt[t, 1]) * (oracle.dequantize(*experts[int(ids[t, 1])][2:4]) @ h[t, 1])
                        for t in range(w.T)])
    assert close(y - y0, contrib, 1e-12)
    # and an out-of-range id in that slot behaves like a zero weight
    ids_bad = ids.copy(); ids_bad[:, 1] = w.E + 5
    h_bad, _ = oracle.gate_up(x, ids_bad, experts, w.E, w.I)
    assert np.all(h_bad[:, 1] == 0)
    assert close(oracle.down(h, ids_bad, wt, experts, w.E, w.H), y0, 1e-14)


def test_topk_order_does_not_matter(mid_case):
    w, x, ids, wt, experts = mid_case
    y = oracle.layer(x, ids, wt, experts, w.E, w.H, w.I)["y_spec"]
    perm = [2, 0, 1]
    yp = oracle.layer(x, ids[:, perm], wt[:, perm], experts, w.E, w.H, w.I)["y_spec"]
    assert close(y, yp, 1e-13)


def test_one_hot_x_selects_a_column(mid_case):
    w, _, ids, wt, experts = mid_case
    for c in [0, 31, 32, 63]:
        x = np.zeros((w.T, w.H)); x[:, c] = 1.0
        _, hp = oracle.gate_up(x, ids, experts, w.E, w.I)
        for t in range(w.T):
            for j in range(w.k):
                wgu, sgu = experts[int(ids[t, j])][:2]
                col_g = [_w(wgu, sgu, i, c) for i in range(w.I)]
                col_u = [_w(wgu, sgu, w.I + i, c) for i in range(w.I)]
                want = [_silu(g) * u for g, u in zip(col_g, col_u)]
                # g and u are single exact products; only exp() may differ in the last ulp
                assert np.allclose(hp[t, j], want, rtol=1e-14, atol=0)


def test_one_hot_h_selects_a_down_column(mid_case):
    w, _, ids, wt, experts = mid_case
    for c in [0, 33, 95]:
        h = np.zeros((w.T, w.k, w.I)); h[:, 2, c] = 1.0
        y = oracle.down(h, ids, wt, experts, w.E, w.H)
        for t in range(w.T):
            wd, sd = experts[int(ids[t, 2])][2:4]
            want = [float(wt[t, 2]) * _w(wd, sd, r, c) for r in range(w.H)]
            assert np.array_equal(y[t], want)


def test_token_permutation_and_batch_consistency(mid_case):
    w, x, ids, wt, experts = mid_case
    y = oracle.layer(x, ids, wt, experts, w.E, w.H, w.I)["y_spec"]
    perm = np.array([3, 1, 0, 2])
    yp = oracle.layer(x[perm], ids[perm], wt[perm], experts, w.E, w.H, w.I)["y_spec"]
    assert np.array_equal(yp, y[perm])
    for t in range(w.T):
        y1 = oracle.layer(x[t:t + 1], ids[t:t + 1], wt[t:t + 1], experts, w.E, w.H, w.I)["y_spec"]
        assert np.array_equal(y1[0], y[t])


def test_duplicate_ids_merge(mid_case):
    w, x, ids, wt, experts = mid_case
    a = int(ids[0, 0])
    ids2 = np.array([[a, a]], np.int32)
    w2 = np.array([[0.25, 0.5]], np.float32)
    h2, _ = oracle.gate_up(x[:1], ids2, experts, w.E, w.I)
    assert np.array_equal(h2[0, 0], h2[0, 1])
    y2 = oracle.down(h2, ids2, w2, experts, w.E, w.H)
    y1 = oracle.down(h2[:, :1], ids2[:, :1], np.array([[0.75]], np.float32), experts, w.E, w.H)
    assert close(y2, y1, 1e-14)


def test_linear_in_routing_weights(mid_case):
    w, x, ids, wt, experts = mid_case
    h, _ = oracle.gate_up(x, ids, experts, w.E, w.I)
    rng = np.random.default_rng(5)
    w1 = rng.random(wt.shape).astype(np.float32)
    w2 = rng.random(wt.shape).astype(np.float32)
    y1 = oracle.down(h, ids, w1, experts, w.E, w.H)
    y2 = oracle.down(h, ids, w2, experts, w.E, w.H)
    y12 = oracle.down(h, ids, (w1.astype(np.float64) + w2).astype(np.float32), experts, w.E, w.H)
    exact = (w1.astype(np.float64) + w2) == (w1 + w2).astype(np.float64)
    if exact.all():
        assert close(y12, y1 + y2, 1e-13)
    y_half = oracle.down(h, ids, w1 / np.float32(2), experts, w.E, w.H)
    assert np.array_equal(y_half * 2, y1)


def test_row_subset_matches_full(mid_case):
    w, x, ids, wt, experts = mid_case
    h, _ = oracle.gate_up(x, ids, experts, w.E, w.I)
    y = oracle.down(h, ids, wt, experts, w.E, w.H)
    rows = np.array([0, 5, 63])
    assert np.array_equal(oracle.down(h, ids, wt, experts, w.E, w.H, rows=rows), y[:, rows])


# ---------------------------------------------------------------------------
# the classic path's MXFP8 requantisation (accuracy comparison only)
# ---------------------------------------------------------------------------

def test_requantize_keeps_representable_blocks():
    rng = np.random.default_rng(21)
    codes = rng.integers(0, 0x7F, size=(8, 64))
    codes[:, 0] = 0x70          # a block max with magnitude 256, so the chosen exponent is exact
    codes[:, 32] = 0x7A         # 384
    vals = oracle.E4M3[codes] * np.where(rng.random((8, 64)) < 0.5, -1, 1)
    e = rng.integers(-20, 5, size=(8, 2))
    a = vals * np.repeat(2.0 ** e, 32, axis=1)
    assert np.array_equal(oracle.requantize_mxfp8(a), a)


def test_requantize_rounding_matches_torch_cast():
    rng = np.random.default_rng(22)
    q = (rng.standard_normal(200000) * 100).astype(np.float32)
    q = np.clip(q, -448, 448)
    want = torch.from_numpy(q).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = om._round_e4m3(q.astype(np.float64))
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# mutation tests: plant a mistake in the oracle, a pin must catch it
# ---------------------------------------------------------------------------

def _brute_agrees():
    w, x, ids, wt, experts = tiny_case(2, 2, 64, 32, 2, seed=314)
    out = oracle.layer(x, ids, wt, experts, w.E, w.H, w.I)
    h_bf, y_bf = brute_layer(x, ids, wt, experts, w.E, w.H, w.I)
    return close(out["h_pure"], h_bf) and close(out["y_pure"], y_bf)


def test_brute_force_catches_planted_mistakes(monkeypatch):
    assert _brute_agrees()
    real_dq = om.dequantize

    def dq_wrong_block(codes, scales):        # scale index K // 16 instead of K // 32
        K = codes.shape[-1]
        s = np.concatenate([np.repeat(oracle.UE8M0[scales], 16, axis=-1)] * 2, axis=-1)[..., :K]
        return oracle.E4M3[codes] * s

    def dq_transposed(codes, scales):
        r = real_dq(codes, scales)
        return r[::-1].copy()

    mutations = [
        ("dequantize", dq_wrong_block),
        ("dequantize", dq_transposed),
        ("silu", lambda z: np.asarray(z) / (1.0 + np.exp(np.asarray(z)))),
    ]
    for name, fn in mutations:
        with monkeypatch.context() as m:
            m.setattr(om, name, fn)
            assert not _brute_agrees(), name


def test_brute_force_catches_swapped_gate_up(monkeypatch):
    real = om.gate_up

    def swapped(x, ids, experts, E, I, tokens=None, fmt="mxfp8"):
        def src(e):
            wgu, sgu, wd, sd = experts[e]
            return (np.concatenate([wgu[I:], wgu[:I]]), np.concatenate([sgu[I:], sgu[:I]]), wd, sd)
        return real(x, ids, src, E, I, tokens=tokens, fmt=fmt)

    monkeypatch.setattr(om, "gate_up", swapped)
    assert not _brute_agrees()


def test_brute_force_catches_misapplied_routing_weight(monkeypatch):
    real = om.down

    def wrong(h, ids, w, experts, E, H, tokens=None, rows=None, fmt="mxfp8"):
        return real(h, ids, np.asarray(w)[:, ::-1].copy(), experts, E, H, tokens=tokens, rows=rows,
                    fmt=fmt)

    monkeypatch.setattr(om, "down", wrong)
    assert not _brute_agrees()
