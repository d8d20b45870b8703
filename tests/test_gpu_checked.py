"""The checked build (libgdn_checked.so, -DGDN_CHECKS): every kernel family on the
smallest shapes (one sequence, one V head) and ragged token counts, in a fresh
process that loads the checked library, with no range check firing (device
error word 0) and results matching the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_runs_every_path_clean():
    from gated_delta_ssm_gb300 import build as gbuild
    gbuild.build()
    env = dict(os.environ, GDN_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "tests._checked_child"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "checked build clean" in r.stdout
