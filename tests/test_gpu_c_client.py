"""The C ABI from a plain C program: tests/c_client/gdn_c_client.c is compiled
against include/gdn.h and libgdn.so (no Python, no torch in the process) and
checks on the GPU that two single-token decode steps and one two-token layer
scan agree bit for bit."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_runs(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    from gated_delta_ssm_gb300 import build as gbuild
    gbuild.build()
    pkg = os.path.join(ROOT, "gated_delta_ssm_gb300")
    exe = tmp_path / "gdn_c_client"
    r = subprocess.run([nvcc, "-o", str(exe), os.path.join(ROOT, "tests", "c_client", "gdn_c_client.c"),
                        "-I", os.path.join(ROOT, "include"), "-L", pkg, "-lgdn",
                        "-Xlinker", "-rpath=" + pkg], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client ok" in r.stdout
