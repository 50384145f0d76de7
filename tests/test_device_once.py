"""The library's one-time launch set-up (a kernel's shared-memory opt-in, the
LM head's resident-pair count) is kept per device: a host-only unit test of
sv::device_once compiled with g++, and a check that no launcher keeps such
state in a process-wide flag."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_42_gb300", "csrc")


def test_device_once_host_logic(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    exe = tmp_path / "device_once_test"
    src = os.path.join(ROOT, "tests", "native", "device_once_test.cpp")
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, src, "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"


def test_no_process_wide_launch_flags():
    """Every cudaFuncSetAttribute and occupancy query sits inside a per-device
    set-up (cuda_once), not behind a static flag shared by all devices."""
    for name in os.listdir(CSRC):
        if not name.endswith((".cu", ".cuh")):
            continue
        with open(os.path.join(CSRC, name)) as f:
            text = f.read()
        assert not re.search(r"static\s+(bool|int)\s+\w+\s*=", text), name
        for m in re.finditer(r"cudaFuncSetAttribute|cudaOccupancyMaxActiveClusters", text):
            head = text[max(0, m.start() - 600):m.start()]
            assert "cuda_once(" in head, (name, text[m.start():m.start() + 60])
