"""Programmatic dependent launch and the deep decode pipeline change only when kernels
start, never what they compute: a mixed scenario (sliding and global layers launched back
to back, decode steps, chunks, resets, a row copy) gives bit-identical outputs and live cache
state (every kept position of every row and layer) with both on (the default) and with both
off (KVINC_PDL=0, KVINC_DEEP=0)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(path, env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(HERE, "pdl_case.py"), path], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return np.load(path)


def test_programmatic_launch_and_deep_pipeline_are_bit_identical(tmp_path):
    on = _run(str(tmp_path / "on.npz"), {"KVINC_PDL": "1", "KVINC_DEEP": "1"})
    off = _run(str(tmp_path / "off.npz"), {"KVINC_PDL": "0", "KVINC_DEEP": "0"})
    assert sorted(on.files) == sorted(off.files) and len(on.files) > 150
    for name in on.files:
        assert np.array_equal(on[name], off[name]), name
