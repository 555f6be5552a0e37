"""Every kernel instance of the library compiles for sm_103a without register spills.

ptxas prints, per entry function, a line "N bytes stack frame, S bytes spill
stores, L bytes spill loads"; this test compiles the library once with
-Xptxas -v (no GPU needed) and requires S = L = 0 for every entry.
"""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

from sparse_expert_gemv_gb300 import build


def ptxas_report():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        cmd = build.command(os.path.join(d, "libcheck.so"), ["-Xptxas", "-v"])
        r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    entries, cur = {}, None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur is not None and cur not in entries:
            entries[cur] = (int(m.group(1)), int(m.group(2)))
    return entries


def test_no_kernel_spills_registers():
    entries = ptxas_report()
    # both formats, KMAX 8 and 32, every token-group size, the one-launch,
    # TMA, MMA and tensor-core kernels
    assert len(entries) >= 60, sorted(entries)
    assert any("moe_layer_fused_t1" in n for n in entries)
    assert any("moe_gate_up_3d_batched_xs" in n for n in entries)
    assert any("moe_down_mma" in n for n in entries)
    spilled = {n: v for n, v in entries.items() if v != (0, 0)}
    assert not spilled, spilled
