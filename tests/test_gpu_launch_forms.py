"""The block backward's outputs do not depend on how its kernels are put on
the GPU: with the weight-gradient side stream and programmatic dependent
launch on the input-gradient chain (the default), with plain stream order
(COLLIDER_PDL=0), and with every launch on the caller's stream
(COLLIDER_SIDE_STREAM=0), every output is bit-identical.  A kernel that read
a buffer before the kernel ahead of it had finished writing it would show up
here.  Each form runs in a child process (the switches are read once per
process)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(tmp_path, name, **env):
    out = os.path.join(str(tmp_path), name + ".npz")
    r = subprocess.run([sys.executable, os.path.join(HERE, "layer_outputs_child.py"), out],
                       env=dict(os.environ, **env), cwd=HERE, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return dict(np.load(out))


def test_outputs_identical_across_launch_forms(tmp_path):
    base = _run(tmp_path, "default")
    for name, env in (("plain_order", {"COLLIDER_PDL": "0"}), ("one_stream", {"COLLIDER_SIDE_STREAM": "0"})):
        got = _run(tmp_path, name, **env)
        assert set(got) == set(base)
        for k in base:
            assert np.array_equal(base[k], got[k]), (name, k)
