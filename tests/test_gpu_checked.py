"""The library built with EXTKV_CHECKED: every plain global load and store
whose index a kernel computes is tested against its buffer first, and an
access outside it is skipped and flagged EXTKV_DEV_BOUNDS in the status word
(device bounds checks in place of a sanitizer, which is closed on this machine:
no trap, no fault).  The GPU test runs every kernel family on that library in
a process of its own against the oracle and requires clean status words; the
CPU test compiles one translation unit in that mode."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.gpu
def test_checked_build_runs_every_kernel_family_without_a_bounds_flag():
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_run.py")], capture_output=True, text=True,
                       timeout=1800, cwd=ROOT)
    assert r.returncode == 0, (r.stdout[-3000:] + r.stderr[-3000:])
    assert "checked ok" in r.stdout, r.stdout[-2000:]


def test_checked_mode_compiles(tmp_path):
    from biased_gqa_attention_gb300 import build
    src = os.path.join(build.CSRC, "scatter_bias.cu")
    cmd = [build._nvcc(), *build.ARCH, *build.NVCC_FLAGS, "-DEXTKV_CHECKED", "-c", src, "-o",
           str(tmp_path / "scatter_bias_checked.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
