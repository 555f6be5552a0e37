"""The C ABI on a machine without a GPU: the library loads, exports every entry
point include/moe_decode.h declares, and rejects bad arguments on the host
before touching CUDA (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_decode.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    b = __graft_entry__._build_module()
    csrc = os.path.join(b.HERE, "csrc")
    newest = max(os.path.getmtime(os.path.join(csrc, f)) for f in os.listdir(csrc))
    if not os.path.exists(b.OUT) or os.path.getmtime(b.OUT) < newest:
        b.build()
    from sparse_expert_gemv_gb300 import _lib
    return _lib.lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_documented_calls():
    names = declared_functions()
    for n in ["moe_decode_create", "moe_decode_destroy", "moe_gate_up", "moe_down", "moe_route",
              "moe_decode_layer", "moe_decode_forward_host", "moe_dedup_schedule",
              "moe_decode_get_error", "moe_status_string", "moe_decode_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from sparse_expert_gemv_gb300 import _lib
    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_status_strings_and_version(lib):
    assert lib.moe_decode_version() == 100
    for s, txt in [(0, b"ok"), (1, b"invalid argument"), (2, b"unsupported shape"),
                   (3, b"misaligned pointer"), (4, b"CUDA runtime error"),
                   (5, b"device flagged an error"), (77, b"unknown status")]:
        assert lib.moe_status_string(s) == txt


def _create(lib, E=8, k=2, H=256, I=128, max_T=4, flags=0, ptrs=(256, 512, 1024, 2048)):
    from sparse_expert_gemv_gb300 import MoEConfig
    cfg = MoEConfig(E, k, H, I, max_T, flags)
    out = ctypes.c_void_p(123)
    st = lib.moe_decode_create(ctypes.byref(cfg), *[ctypes.c_void_p(p) for p in ptrs],
                               ctypes.byref(out))
    return st, out.value


@pytest.mark.parametrize("kw,status", [
    (dict(E=0), 1), (dict(k=0), 1), (dict(k=9, E=8), 1), (dict(H=0), 1), (dict(max_T=-1), 1),
    (dict(H=48), 2), (dict(I=100), 2), (dict(E=2048, k=2), 2), (dict(k=33, E=64), 2),
    (dict(k=32, E=64, I=2048), 2),                    # k*I*4 bytes of h exceed shared memory
    (dict(flags=0x80), 1),
    (dict(ptrs=(0, 512, 1024, 2048)), 1), (dict(ptrs=(256, 0, 1024, 2048)), 1),
    (dict(ptrs=(256 + 16, 512, 1024, 2048)), 3), (dict(ptrs=(256, 512, 1024 + 8, 2048)), 3),
])
def test_create_rejects_bad_arguments_without_cuda(lib, kw, status):
    st, h = _create(lib, **kw)
    assert st == status
    assert h is None


def test_null_handle_and_null_config(lib):
    assert lib.moe_decode_create(None, None, None, None, None, None) == 1
    z = ctypes.c_void_p(0)
    assert lib.moe_gate_up(None, 1, z, z, z, z) == 1
    assert lib.moe_down(None, 1, z, z, z, z, z) == 1
    assert lib.moe_route(None, 1, z, z, z, z) == 1
    assert lib.moe_decode_layer(None, 1, z, z, z, z, z, z) == 1
    assert lib.moe_decode_forward_host(None, 1, z, z, z, z, z) == 1
    assert lib.moe_dedup_schedule(None, 1, z, z, z, z, z, z) == 1
    assert lib.moe_decode_get_error(None, None) == 1
    assert lib.moe_decode_get_error_stream(None, None, None) == 1
    assert lib.moe_decode_destroy(None) == 0
    assert lib.moe_decode_kernel_name(None, 1, 0) == b""


def test_timeline_library_exports_its_header():
    # the MOE_TIMELINE build exports every call of both headers
    import __graft_entry__
    b = __graft_entry__._build_module()
    if b.stale(b.OUT_TIMELINE):
        b.build(timeline=True)
    tl = ctypes.CDLL(b.OUT_TIMELINE)
    text = open(os.path.join(ROOT, "include", "moe_decode_timeline.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))
    assert "moe_decode_layer_timeline" in names
    for n in names + declared_functions():
        assert hasattr(tl, n), n
    tl.moe_decode_timeline_ctas.argtypes = [ctypes.c_void_p]
    assert tl.moe_decode_timeline_ctas(None) == -1
