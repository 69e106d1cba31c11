"""Child process of test_gpu_launch_forms: one filtered backward of a block
with several key and query blocks per sequence, its outputs saved to the .npz
named on the command line.  The launch switches (COLLIDER_PDL,
COLLIDER_SIDE_STREAM) come from the environment, which the library reads once
per process."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import workloads  # noqa: E402
from oracle import block as ob  # noqa: E402
import gpu_util as gu  # noqa: E402


def main(path: str) -> None:
    s = workloads.LayerShape(seed_base=84000, arch="llama", B=2, T=1100, D=256, H=4, Hkv=2, dh=64, F=384,
                             rotary_dim=64, rope_base=10000.0, norm="rms", eps=1e-5, act="swiglu",
                             qkv_bias=False, out_bias=False, mlp_bias=False, f=0.4, mask="gumbel")
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    _, saved = ob.block_forward(t["x"], w, s, round_saved=True)
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    out = L.results()
    gu.cl.collider_check()
    np.savez(path, **out)


if __name__ == "__main__":
    main(sys.argv[1])
