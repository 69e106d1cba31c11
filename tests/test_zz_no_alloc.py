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


def _noalloc(keep, stream=None):
    B, T = keep.shape
    mask = torch.from_numpy(np.ascontiguousarray(keep)).to(gu.DEV)
    idx = torch.full((B * T,), -1, dtype=torch.int32, device=gu.DEV)
    cu = torch.full((B + 1,), -1, dtype=torch.int32, device=gu.DEV)
    nk = torch.full((1,), -1, dtype=torch.int32, device=gu.DEV)
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())   # the inputs above are ready
    cl.collider_compact_noalloc(mask, B, T, idx, cu, nk, stream)
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


def test_honours_its_stream():
    """Work goes on the stream it is given: a side stream, behind a long
    kernel queued there first, still gives collider_compact's bits."""
    rng = np.random.default_rng(7)
    keep = (rng.random((2, 300_000)) >= 0.35).astype(np.uint8)
    side = torch.cuda.Stream()
    busy = torch.empty(64 << 20, dtype=torch.float32, device=gu.DEV)
    with torch.cuda.stream(side):
        busy.normal_()            # keeps the side stream busy while the call is queued behind it
    a = _noalloc(keep, side)
    b = gu.compact(keep)
    side.synchronize()
    torch.cuda.synchronize()
    n = int(b[2].item())
    assert int(a[2].item()) == n
    assert torch.equal(a[0][:n], b[0][:n]) and torch.equal(a[1], b[1])
    cl.collider_check()


def test_exactly_at_its_limit():
    """2^30 tokens (65,536 sequences of 16,384): every one of the array's
    65,536 per-chunk counts is used.  A few tokens are kept; the index list,
    the per-sequence offsets and the count must come out exact."""
    B, T = 1 << 16, 1 << 14
    M = B * T
    kept = np.array([0, 16_383, 16_384, 123_456_789, 700_000_001, M - 16_385, M - 1], dtype=np.int64)
    mask = torch.zeros(M, dtype=torch.uint8, device=gu.DEV)
    mask[torch.from_numpy(kept).to(gu.DEV)] = 1
    idx = torch.full((M,), -1, dtype=torch.int32, device=gu.DEV)
    cu = torch.full((B + 1,), -1, dtype=torch.int32, device=gu.DEV)
    nk = torch.full((1,), -1, dtype=torch.int32, device=gu.DEV)
    cl.collider_compact_noalloc(mask, B, T, idx, cu, nk)
    torch.cuda.synchronize()
    cl.collider_check()
    assert int(nk.item()) == kept.size
    assert np.array_equal(idx[:kept.size].cpu().numpy(), kept.astype(np.int32))
    per_seq = np.bincount(kept // T, minlength=B)
    want_cu = np.concatenate([[0], np.cumsum(per_seq)]).astype(np.int32)
    assert np.array_equal(cu.cpu().numpy(), want_cu)
    assert int(idx[kept.size]) == -1          # nothing written past n_kept
    del mask, idx
    torch.cuda.empty_cache()
