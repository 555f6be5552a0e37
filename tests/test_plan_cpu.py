"""Host-side launch planning, without a GPU (moe_decode_plan): the one-launch
single-token layer's ring, the several-token kernels' choices, token groups
and shared-memory budgets, checked against the rules the kernels rely on
(shared-memory limits, TMA alignment, whole K-chunks and row granules)
over a sweep of shapes, and the choices for the seeded workloads."""
import ctypes
import itertools

import pytest

import workloads as wl
from sparse_expert_gemv_gb300._lib import MOE_FLAG_MXFP4, MOE_FLAG_WARP_MMA, MoEConfig, MoEPlan, lib

SMS, SMEM = 152, 232448          # GB300: SMs and opt-in shared memory per CTA


def plan(E, k, H, I, T, fmt="mxfp8", sms=SMS, smem=SMEM, flags=0):
    cfg = MoEConfig(E, k, H, I, T, (MOE_FLAG_MXFP4 if fmt == "mxfp4" else 0) | flags)
    out = MoEPlan()
    st = lib.moe_decode_plan(ctypes.byref(cfg), sms, smem, T, ctypes.byref(out))
    return st, out


def test_plan_rejects_what_create_rejects():
    assert plan(8, 2, 48, 128, 1)[0] == 2            # H not a multiple of 32
    assert plan(8, 9, 256, 128, 1)[0] == 1           # k > E
    assert plan(8, 2, 256, 128, 0)[0] == 1           # T < 1
    assert plan(8, 2, 256, 128, 1, sms=0)[0] == 1
    assert lib.moe_decode_plan(None, SMS, SMEM, 1, None) == 1


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_seeded_workloads(fmt):
    # the warp path's kernels (workload 3's layer takes the tensor-core path
    # when the weights allow it); with MOE_FLAG_WARP_MMA the 32-token
    # workload's take the warp-level MMA
    want_gu = {0: 0, 1: 0, 2: 1, 3: 1, 4: 1}      # 0 L1, 1 x staged, 2 TMA + mma
    want_dn = {0: 0, 1: 0, 2: 1, 3: 1, 4: 1}      # 0 warp per output, 1 TMA, 2 TMA + mma
    for c, w in wl.WORKLOADS.items():
        st, p = plan(w.E, w.k, w.H, w.I, w.T, fmt)
        assert st == 0
        assert p.gate_up_kernel == want_gu[c], (c, fmt)
        assert p.down_kernel == want_dn[c], (c, fmt)
        assert p.fused == (0 if c == 0 else 1), (c, fmt)
        st, p = plan(w.E, w.k, w.H, w.I, w.T, fmt, flags=MOE_FLAG_WARP_MMA)
        assert (p.gate_up_kernel, p.down_kernel) == ((2, 2) if c == 3 else (want_gu[c], want_dn[c]))
    # the large-expert workload's gate/up runs as two groups of 8 tokens
    w = wl.workload(4)
    assert plan(w.E, w.k, w.H, w.I, w.T, fmt)[1].gate_up_group == 8


SHAPES = list(itertools.product([8, 128, 256], [1, 2, 8, 32], [256, 512, 1024, 2048, 2560, 7168],
                                [32, 96, 128, 384, 768, 2048], [1, 2, 8, 16, 32, 40]))


@pytest.mark.parametrize("mma", [False, True])
@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_plan_invariants_over_shapes(fmt, mma):
    cb = 16 if fmt == "mxfp4" else 32               # code bytes per 32-element block
    n = 0
    for E, k, H, I, T in SHAPES:
        if k > E:
            continue
        st, p = plan(E, k, H, I, T, fmt, flags=MOE_FLAG_WARP_MMA if mma else 0)
        if not mma:
            assert p.gate_up_kernel != 2 and p.down_kernel != 2
        assert st == 0
        n += 1
        if p.fused:
            # shared memory, whole K-chunks, 128-byte slots, a chunk's down
            # groups all resident, row chunks of whole 16-byte-aligned granules
            assert p.fused_smem <= SMEM
            assert H % p.fused_kc == 0 and H % 512 == 0 and I % 128 == 0
            assert p.fused_slot_bytes % 128 == 0
            assert p.fused_down_per_slot >= 1 and -(-k // p.fused_down_per_slot) <= p.fused_slots
            nbI = I // 32
            assert (p.fused_down_rows * nbI) % 16 == 0 and 1 <= p.fused_down_rows <= 15
            assert (p.fused_down_rows * I * cb // 32) % 128 == 0   # scale copy destination
        assert 1 <= p.gate_up_group <= min(T, 32)
        if p.gate_up_kernel == 2:
            assert p.gate_up_group >= 16 and 2 <= p.gate_up_slots <= 16
            assert p.gate_up_smem <= SMEM and H % (512 * 32 // cb) == 0
        if p.gate_up_kernel == 1:
            assert p.gate_up_group >= 2 and p.gate_up_smem <= SMEM
        if p.down_kernel:
            assert I % 128 == 0 and I <= 2048 and p.down_smem <= SMEM and p.down_slots >= 2
            assert (16 * (I // 32)) % 16 == 0       # a tile's scale bytes: whole 16-byte units
        if p.down_kernel == 2:
            assert min(T, 32) >= 16 and I * cb // 32 <= 1024 and 6 <= p.down_slots <= 16
    assert n > 500
