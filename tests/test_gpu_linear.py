"""GPU parity: linear backward, f32 (single linear layer workload, f32 FMA) and
bf16 (tcgen05 GEMMs), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import workloads
from oracle import ops

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
cl = gu.cl


def _run(dtype, X, W, dY, keep, x_rows, dy_rows, dx_rows, want_db=True):
    M, K = X.shape
    N = W.shape[1]
    idx, cu, nk = gu.compact(keep.reshape(1, -1))
    n = int(keep.sum())
    kept = np.flatnonzero(keep.reshape(-1))
    up = gu.f32 if dtype == cl.F32 else gu.bf16
    Xd = up(X if x_rows == cl.ROWS_FULL else np.vstack([X[kept], np.zeros((M - n, K))]))
    dYd = up(dY if dy_rows == cl.ROWS_FULL else np.vstack([dY[kept], np.zeros((M - n, N))]))
    Wd = up(W)
    tdt = torch.float32 if dtype == cl.F32 else torch.bfloat16
    dX = torch.full((M, K), float("nan"), dtype=tdt, device=gu.DEV)
    dW = torch.full((K, N), float("nan"), dtype=torch.float32, device=gu.DEV)
    db = torch.full((N,), float("nan"), dtype=torch.float32, device=gu.DEV) if want_db else None
    ws = torch.empty(max(cl.collider_linear_workspace_size(dtype, M, K, N), 1), dtype=torch.uint8, device=gu.DEV)
    cl.collider_linear_bwd(dtype, M, K, N, Xd, x_rows, Wd, dYd, dy_rows, idx, nk, dX, dx_rows, dW, db, ws)
    cl.collider_check()
    rX, rW, rb = ops.linear_backward(gu.host(up(X)), gu.host(Wd), gu.host(up(dY)), keep.reshape(-1) != 0,
                                     want_bias=True)
    gX = gu.host(dX)
    if dx_rows == cl.ROWS_COMPACT:
        gX, rX = gX[:n], rX[kept]
        pad = min(-(-n // 128) * 128, M)
        assert np.all(gu.host(dX)[n:pad] == 0)
    return (gX, rX), (gu.host(dW), rW), ((gu.host(db), rb) if want_db else None)


def test_single_linear_workload_f32():
    s = workloads.WORKLOADS["linear_fp32"]
    t = workloads.linear_inputs(s)
    keep = t["keep"].reshape(-1)
    assert keep.sum() == 77
    (gX, rX), (gW, rW), (gb, rb) = _run(cl.F32, t["X"], t["W"], t["dY"], keep, cl.ROWS_FULL, cl.ROWS_FULL,
                                        cl.ROWS_FULL)
    assert gu.rel_err(gX, rX) <= 1e-4
    assert gu.rel_err(gW, rW) <= 1e-4
    assert gu.rel_err(gb, rb) <= 1e-4
    assert np.all(gX[keep == 0] == 0)


@pytest.mark.parametrize("rows", [(cl.ROWS_COMPACT, cl.ROWS_COMPACT, cl.ROWS_COMPACT),
                                  (cl.ROWS_FULL, cl.ROWS_COMPACT, cl.ROWS_FULL)])
def test_f32_row_layouts(rows):
    rng = np.random.default_rng(1)
    M, K, N = 300, 72, 136
    X, W, dY = rng.normal(size=(M, K)), rng.normal(size=(K, N)) / 8, rng.normal(size=(M, N))
    keep = (rng.random(M) < 0.55).astype(np.uint8)
    for g, r in _run(cl.F32, X, W, dY, keep, *rows):
        assert gu.rel_err(g, r) <= 1e-4


@pytest.mark.parametrize("M,K,N,f", [(4096, 2048, 5632, 0.4),    # MLP down-projection shape, 1 sequence
                                     (1000, 200, 328, 0.3),      # ragged: not tile multiples
                                     (257, 64, 512, 0.0),
                                     (640, 512, 256, 0.9)])
def test_bf16_tcgen05_gemms(M, K, N, f):
    rng = np.random.default_rng(M + K + N)
    X = workloads.bf16_representable(rng.normal(size=(M, K)))
    W = workloads.bf16_representable(rng.normal(size=(K, N)) * 0.02)
    dY = workloads.bf16_representable(rng.normal(size=(M, N)))
    keep = workloads.gumbel_keep_mask(1, M, f, seed=M).reshape(-1)
    for g, r in _run(cl.BF16, X, W, dY, keep, cl.ROWS_FULL, cl.ROWS_FULL, cl.ROWS_FULL):
        assert gu.rel_err(g, r) <= 2e-2


def test_bf16_compact_layouts_and_empty():
    rng = np.random.default_rng(7)
    M, K, N = 384, 128, 256
    X = workloads.bf16_representable(rng.normal(size=(M, K)))
    W = workloads.bf16_representable(rng.normal(size=(K, N)) * 0.05)
    dY = workloads.bf16_representable(rng.normal(size=(M, N)))
    keep = (rng.random(M) < 0.5).astype(np.uint8)
    for g, r in _run(cl.BF16, X, W, dY, keep, cl.ROWS_COMPACT, cl.ROWS_COMPACT, cl.ROWS_COMPACT):
        assert gu.rel_err(g, r) <= 2e-2
    # nothing kept: every gradient exactly zero
    for g, r in _run(cl.BF16, X, W, dY, np.zeros(M, np.uint8), cl.ROWS_FULL, cl.ROWS_FULL, cl.ROWS_FULL):
        assert np.all(g == 0)
    # NaN in filtered rows of the inputs cannot leak
    keep = (rng.random(M) < 0.5).astype(np.uint8)
    Xn, dYn = X.copy(), dY.copy()
    Xn[keep == 0] = np.nan
    dYn[keep == 0] = np.inf
    a = _run(cl.BF16, X, W, dY, keep, cl.ROWS_FULL, cl.ROWS_FULL, cl.ROWS_FULL)
    b = _run(cl.BF16, Xn, W, dYn, keep, cl.ROWS_FULL, cl.ROWS_FULL, cl.ROWS_FULL)
    for (ga, _), (gb, _) in zip(a, b):
        assert np.array_equal(ga, gb)


def test_bf16_dw_is_deterministic():
    rng = np.random.default_rng(8)
    M, K, N = 2048, 256, 512
    X = workloads.bf16_representable(rng.normal(size=(M, K)))
    W = workloads.bf16_representable(rng.normal(size=(K, N)) * 0.05)
    dY = workloads.bf16_representable(rng.normal(size=(M, N)))
    keep = (rng.random(M) < 0.6).astype(np.uint8)
    a = _run(cl.BF16, X, W, dY, keep, cl.ROWS_FULL, cl.ROWS_FULL, cl.ROWS_FULL)
    b = _run(cl.BF16, X, W, dY, keep, cl.ROWS_FULL, cl.ROWS_FULL, cl.ROWS_FULL)
    for (ga, _), (gb, _) in zip(a, b):
        assert np.array_equal(ga, gb)
