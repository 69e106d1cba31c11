"""GPU parity of the tcgen05 GEMM in its other launch form.  Whole-tile GEMM
launches with 256-wide tiles normally run as 2-SM CTA pairs (each CTA loads only
its own tiles; no copy is multicast); 128-wide tiles and stream-K launches run
as lone CTAs.  COLLIDER_GEMM_PAIR=0 makes every launch a lone CTA.  The
library reads the switch once per process, so the linear-layer and block
parity tests run again in a child process with it set."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_linear_and_block_parity_with_lone_ctas():
    env = dict(os.environ, COLLIDER_GEMM_PAIR="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_gpu_linear.py"), os.path.join(HERE, "test_gpu_layer.py")],
                       env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
