"""The single-kernel backward (head dims 72..128, selected with
FATTN_BWD_FUSED=1): the backward parity tests of test_gpu_backward.py and
the head-dim backward tests, re-run in a child process with the switch set
(the library reads it once per process), against the same fp64 oracle and
bars."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fused_backward_parity(cuda_device):
    env = dict(os.environ, FATTN_BWD_FUSED="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
         "tests/test_gpu_backward.py", "tests/test_gpu_headdim.py", "-k", "backward"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    tail = "\n".join((r.stdout + r.stderr).strip().splitlines()[-15:])
    assert r.returncode == 0, f"fused backward parity failed:\n{tail}"
    assert " passed" in tail, tail
