"""The bench's recorded ncu traffic applies only to the code it was taken from.

bench.source_hash() hashes the one-launch kernel's sources with comments and
blank lines removed: a comment edit keeps a recorded figure valid, any code
edit voids it (recorded_traffic() then returns None).
"""
import json
import os
import shutil

import bench


def _copy_sources(tmp_path):
    for f in bench.FUSED_SOURCES:
        dst = tmp_path / f
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copyfile(os.path.join(bench.ROOT, f), dst)


def _append(path, text):
    with open(path, "a") as fh:
        fh.write(text)


def test_hash_ignores_comments_and_sees_code(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash()
    kernel = tmp_path / "sparse_expert_gemv_gb300/csrc/moe_layer_fused.cuh"
    _append(kernel, "\n// a note\n/* a block\n   comment */\n\n")
    assert bench.source_hash() == h0
    _append(kernel, "static_assert(true, \"x\");\n")
    assert bench.source_hash() != h0


def test_recorded_traffic_needs_a_matching_hash(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    kernel, workload, fmt = "moe_layer_fused_t1", "batch-1 decode E128 k8 H2048 I768 T1", "mxfp8"
    (tmp_path / "profiles").mkdir()
    rec = {bench.traffic_key(kernel, workload, fmt): {
        "source_hash": bench.source_hash(), "dram_bytes_per_launch_full": 1234.0}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic(kernel, workload, fmt) == 1234.0
    assert bench.recorded_traffic(kernel, workload, "mxfp4") is None
    _append(tmp_path / "sparse_expert_gemv_gb300/csrc/moe_decode.cu", "int moe_changed_code = 1;\n")
    assert bench.recorded_traffic(kernel, workload, fmt) is None
