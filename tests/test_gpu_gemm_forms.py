"""GPU parity of the tcgen05 GEMM in its other launch forms.  Whole-tile GEMM
launches normally run as CTA pairs: 2-SM MMAs for 256-wide tiles, B-tile
multicast for 128-wide ones.  COLLIDER_GEMM_PAIR=0 makes them run as lone CTAs,
COLLIDER_GEMM_PAIR=1 as multicast pairs everywhere.  The library reads the
switch once per process, so the linear-layer and block parity tests run again
in a child process with it set."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("form", ["0", "1"])
def test_linear_and_block_parity_in_other_gemm_forms(form):
    env = dict(os.environ, COLLIDER_GEMM_PAIR=form)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_gpu_linear.py"), os.path.join(HERE, "test_gpu_layer.py")],
                       env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
