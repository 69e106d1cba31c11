"""GPU parity: compaction (bit-exact against the oracle) and row gather /
scatter (bit-exact against numpy indexing)."""
import numpy as np
import pytest
import torch

import workloads
from oracle.compaction import compact as oracle_compact

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
cl = gu.cl


def _check(keep):
    idx, cu, nk = gu.compact(keep)
    ri, rc, rn = oracle_compact(keep)
    torch.cuda.synchronize()
    assert int(nk.item()) == rn
    assert np.array_equal(idx[:rn].cpu().numpy(), ri)
    assert np.array_equal(cu.cpu().numpy(), rc)
    assert np.all(idx[rn:].cpu().numpy() == -1)      # nothing written past n_kept


@pytest.mark.parametrize("name", ["linear_fp32", "tinyllama_layer", "qwen25_layer", "phi15_layer"])
def test_workload_masks(name):
    s = workloads.WORKLOADS[name]
    for f in ((0.0, 0.2, 0.4, 0.6) if name == "phi15_layer" else (s.f,)):
        _check(workloads.keep_mask(s.B, s.T, f, s.mask, s.seed_base))


def test_stack_mask_long_sequence():
    s = workloads.WORKLOADS["tinyllama_stack"].layer
    _check(workloads.keep_mask(s.B, s.T, s.f, s.mask, 5000))


@pytest.mark.parametrize("B,T", [(1, 1), (3, 7), (5, 33), (2, 1000), (7, 4099), (1, 16385)])
def test_ragged_and_edges(B, T):
    rng = np.random.default_rng(B * 1000 + T)
    _check((rng.random((B, T)) < 0.5).astype(np.uint8))
    _check(np.zeros((B, T), np.uint8))
    _check(np.ones((B, T), np.uint8))
    _check((rng.integers(0, 256, size=(B, T))).astype(np.uint8))   # any nonzero byte keeps


def test_multi_block_path():
    # above 2^22 tokens the library scans the mask with three kernels
    B, T = 3, 1_500_001
    rng = np.random.default_rng(3)
    _check((rng.random((B, T)) < 0.6).astype(np.uint8))


def test_unaligned_mask_pointer():
    rng = np.random.default_rng(4)
    keep = (rng.random((4, 77)) < 0.5).astype(np.uint8)
    buf = torch.zeros(4 * 77 + 1, dtype=torch.uint8, device=gu.DEV)
    buf[1:] = torch.from_numpy(keep.reshape(-1)).to(gu.DEV)
    idx = torch.full((4 * 77,), -1, dtype=torch.int32, device=gu.DEV)
    cu = torch.zeros(5, dtype=torch.int32, device=gu.DEV)
    nk = torch.zeros(1, dtype=torch.int32, device=gu.DEV)
    cl.collider_compact(buf.data_ptr() + 1, 4, 77, idx, cu, nk)
    ri, rc, rn = oracle_compact(keep)
    torch.cuda.synchronize()
    assert int(nk.item()) == rn and np.array_equal(idx[:rn].cpu().numpy(), ri)
    assert np.array_equal(cu.cpu().numpy(), rc)


@pytest.mark.parametrize("M,row_bytes,f", [(300, 48, 0.4), (1000, 4096, 0.3), (129, 16, 0.0), (64, 32, 1.0)])
def test_gather_scatter(M, row_bytes, f):
    rng = np.random.default_rng(M)
    keep = (rng.random((1, M)) >= f).astype(np.uint8)
    idx, cu, nk = gu.compact(keep)
    n = int(keep.sum())
    src = torch.from_numpy(rng.integers(0, 256, size=(M, row_bytes), dtype=np.uint8)).to(gu.DEV)
    dst = torch.full((M, row_bytes), 0xAB, dtype=torch.uint8, device=gu.DEV)
    cl.collider_gather_rows(src, row_bytes, dst, row_bytes, row_bytes, M, idx, nk)
    torch.cuda.synchronize()
    kept = np.flatnonzero(keep.reshape(-1))
    d = dst.cpu().numpy()
    assert np.array_equal(d[:n], src.cpu().numpy()[kept])
    pad = min(-(-n // 128) * 128, M)
    assert np.all(d[n:pad] == 0) and np.all(d[pad:] == 0xAB)
    full = torch.full((M, row_bytes), 0xCD, dtype=torch.uint8, device=gu.DEV)
    cl.collider_scatter_rows(dst, row_bytes, full, row_bytes, row_bytes, M, idx, nk)
    torch.cuda.synchronize()
    want = np.zeros((M, row_bytes), np.uint8)
    want[kept] = src.cpu().numpy()[kept]
    assert np.array_equal(full.cpu().numpy(), want)


def test_argument_errors_are_reported():
    with pytest.raises(cl.ColliderError, match="INVALID_ARG"):
        cl.collider_compact(None, 1, 4, None, None, None)
    t = torch.zeros(64, dtype=torch.uint8, device=gu.DEV)
    with pytest.raises(cl.ColliderError, match="INVALID_ARG"):
        cl.collider_gather_rows(t, 16, t, 16, 8, 4, t, t)     # row_bytes not a multiple of 16
    cl.collider_check()


@pytest.mark.parametrize("B,T,n", [(4, 2048, 819), (1, 8192, 3276), (3, 100, 0), (3, 100, 100), (2, 5000, 1),
                                   (5, 33, 17)])
def test_select_keep_matches_oracle(B, T, n):
    from oracle.compaction import select_keep
    rng = np.random.default_rng(B * T + n)
    s = rng.gumbel(size=(B, T)).astype(np.float32)
    s[:, ::7] = np.round(s[:, ::7])                 # plenty of ties
    s[0, 3 % T] = np.nan
    s[-1, 5 % T] = -0.0
    s[-1, 6 % T] = 0.0
    s[0, 1 % T] = -np.inf
    mask = torch.full((B, T), 7, dtype=torch.uint8, device=gu.DEV)
    cl.collider_select_keep(torch.from_numpy(s).to(gu.DEV), B, T, n, mask)
    torch.cuda.synchronize()
    assert np.array_equal(mask.cpu().numpy(), select_keep(s, n))
    # scores -> mask -> kept-index list, end to end on the device
    idx, cu, nk = gu.compact(mask.cpu().numpy())
    ri, rc, rn = oracle_compact(select_keep(s, n))
    assert int(nk.item()) == rn and np.array_equal(idx[:rn].cpu().numpy(), ri)
