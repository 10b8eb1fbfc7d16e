"""The checked debug build (-DEB_CHECKS, libeb_sampler_checks.so) on the GPU.

The build tests every computed index of the streaming and selection kernels before using it
and records a failed check in a device word instead of trapping.  Its parity runs in a child
process that loads the checked library (EB_SAMPLER_LIB): the same cases as the parity tests,
the full-size single step and a short loop, compared with the oracle, with no check failing.
"""
import os
import subprocess
import sys

import pytest
import torch

import canvas_sampler_step_b300 as eb

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_matches_the_oracle_with_no_failed_check():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eb.build_checks()
    env = dict(os.environ, EB_SAMPLER_LIB=eb.CHECKS_LIB_PATH, EB_TIE_REPORT="")
    out = subprocess.run([sys.executable, os.path.join(HERE, "checked_build_run.py")], env=env,
                         capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "checked build ok" in out.stdout
