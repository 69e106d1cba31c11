"""collider_compact_noalloc: the compaction entry point that allocates nothing.

Some callers cannot allocate device memory -- programs whose memory is owned
by their own pool allocator, and latency-critical paths where cudaMalloc's
implicit device synchronisation is unacceptable.  This entry point keeps its
scratch in a fixed array inside the library.  Here it is called through the C
ABI and must give the same bits as collider_compact, on two calls in a row
(the shared array keeps the first call's contents, which must not leak into
the second).  Kept in its own file, collected last.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
cl = gu.cl


def _noalloc(keep):
    B, T = keep.shape
    mask = torch.from_numpy(np.ascontiguousarray(keep)).to(gu.DEV)
    idx = torch.full((B * T,), -1, dtype=torch.int32, device=gu.DEV)
    cu = torch.full((B + 1,), -1, dtype=torch.int32, device=gu.DEV)
    nk = torch.full((1,), -1, dtype=torch.int32, device=gu.DEV)
    cl.collider_compact_noalloc(mask, B, T, idx, cu, nk)
    return idx, cu, nk


@pytest.mark.parametrize("B,T,f", [(4, 2048, 0.4), (3, 1000, 0.9), (1, 5_000_003, 0.3)])
def test_matches_collider_compact_twice(B, T, f):
    rng = np.random.default_rng(B * T)
    # two different masks: the second call must not see the first call's counts
    for call, p in enumerate((f, 1.0 - f)):
        keep = (rng.random((B, T)) >= p).astype(np.uint8)
        a = _noalloc(keep)
        b = gu.compact(keep)
        torch.cuda.synchronize()
        n = int(b[2].item())
        assert int(a[2].item()) == n, call
        assert torch.equal(a[0][:n], b[0][:n]), call
        assert torch.equal(a[1], b[1]), call
    cl.collider_check()


def test_rejects_sizes_beyond_its_limit():
    t = torch.zeros(16, dtype=torch.int32, device=gu.DEV)
    with pytest.raises(cl.ColliderError, match="limit"):
        cl.collider_compact_noalloc(t, 1 << 16, (1 << 14) + 1, t, t, t)
