"""GPU parity: filtered attention backward (Figs. 3 and 5) against the fp64
oracle, with and without the RoPE backward, GQA and MHA, head dims 64/128."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import ops
from oracle.attention import attention_forward, filtered_attention_backward

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
cl = gu.cl


def _case(B, T, H, Hkv, dh, f, mask, seed, qk_std=1.0, causal=True):
    rng = np.random.default_rng(seed)
    R = workloads.bf16_representable
    q = R(rng.normal(size=(B * T, H, dh)) * qk_std)
    k = R(rng.normal(size=(B * T, Hkv, dh)) * qk_std)
    v = R(rng.normal(size=(B * T, Hkv, dh)))
    dO = R(rng.normal(size=(B * T, H, dh)))
    keep = workloads.keep_mask(B, T, f, mask, seed)
    scale = 1 / math.sqrt(dh)
    _, lse = attention_forward(q, k, v, B, T, scale, causal=causal)
    lse = lse.astype(np.float32)
    return q, k, v, dO, lse, keep, scale


@pytest.mark.parametrize("B,T,H,Hkv,dh,f,mask,rot", [
    (2, 200, 4, 2, 64, 0.4, "gumbel", 64),     # GQA, ragged sequence lengths
    (1, 300, 2, 1, 128, 0.4, "gumbel", 128),   # head dim 128
    (2, 700, 6, 2, 128, 0.4, "gumbel", 128),   # head dim 128, GQA 3, several 64-query blocks per key block
    (2, 130, 2, 2, 64, 0.6, "span", 32),       # MHA, partial rotary, span mask
    (1, 64, 2, 2, 64, 0.0, "gumbel", 0),       # nothing filtered, no RoPE
    (3, 100, 4, 1, 64, 0.2, "gumbel", 16),
    (1, 1100, 8, 2, 64, 0.3, "gumbel", 64),    # many key / query blocks per sequence
])
@pytest.mark.parametrize("rows", ["full", "compact"])
def test_attention_backward(B, T, H, Hkv, dh, f, mask, rot, rows):
    q, k, v, dO, lse, keep, scale = _case(B, T, H, Hkv, dh, f, mask, seed=T + H + dh, qk_std=1.5)
    M = B * T
    idx, cu, nk = gu.compact(keep)
    n = int(keep.sum())
    kept = np.flatnonzero(keep.reshape(-1))
    full = rows == "full"
    pick = (lambda a: a) if full else (lambda a: np.concatenate([a[kept], np.zeros((M - n,) + a.shape[1:])]))
    Qd, Kd, Vd, dOd = (gu.bf16(pick(a).reshape(M, -1)) for a in (q, k, v, dO))
    dQ = torch.full((M, H * dh), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    dK = torch.full((M, Hkv * dh), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    dV = torch.full((M, Hkv * dh), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    ws = torch.empty(cl.collider_attn_workspace_size(B, T, H, Hkv, dh), dtype=torch.uint8, device=gu.DEV)
    mode = cl.ROWS_FULL if full else cl.ROWS_COMPACT
    cl.collider_attn_bwd(B, T, H, Hkv, dh, 1, scale, rot, 10000.0, Qd, Kd, Vd, None, dOd, H * dh, Hkv * dh,
                         H * dh, mode, gu.f32(lse), idx, cu, nk, dQ, dK, dV, mode, ws)
    cl.collider_check()
    rq, rk, rv = filtered_attention_backward(q, k, v, dO, lse, keep, scale)
    pos = np.tile(np.arange(T), B)
    if rot:
        rq = ops.rope_backward(rq, pos, rot, 10000.0)
        rk = ops.rope_backward(rk, pos, rot, 10000.0)
    for got, ref, nh in ((dQ, rq, H), (dK, rk, Hkv), (dV, rv, Hkv)):
        g = gu.host(got).reshape(M, nh, dh)
        if not full:
            g, ref = g[:n], ref[kept]
            pad = min(-(-n // 128) * 128, M)
            assert np.all(gu.host(got)[n:pad] == 0)
        else:
            assert np.all(g[keep.reshape(-1) == 0] == 0)
        assert gu.rel_err(g, ref) <= 2e-2


def test_attention_ignores_filtered_rows():
    B, T, H, Hkv, dh = 2, 160, 4, 2, 64
    q, k, v, dO, lse, keep, scale = _case(B, T, H, Hkv, dh, 0.4, "gumbel", seed=11)
    M = B * T
    idx, cu, nk = gu.compact(keep)
    km = keep.reshape(-1) == 0
    outs = []
    for poison in (False, True):
        arrs = [a.copy() for a in (q, k, v, dO)]
        l2 = lse.copy()
        if poison:
            for a in arrs:
                a[km] = np.nan
            l2[np.broadcast_to((keep == 0)[:, None, :], l2.shape)] = np.inf
        Qd, Kd, Vd, dOd = (gu.bf16(a.reshape(M, -1)) for a in arrs)
        res = [torch.zeros((M, n * dh), dtype=torch.bfloat16, device=gu.DEV) for n in (H, Hkv, Hkv)]
        ws = torch.empty(cl.collider_attn_workspace_size(B, T, H, Hkv, dh), dtype=torch.uint8, device=gu.DEV)
        cl.collider_attn_bwd(B, T, H, Hkv, dh, 1, scale, 64, 10000.0, Qd, Kd, Vd, None, dOd, H * dh, Hkv * dh,
                             H * dh, cl.ROWS_FULL, gu.f32(l2), idx, cu, nk, *res, cl.ROWS_FULL, ws)
        torch.cuda.synchronize()
        outs.append([r.cpu() for r in res])
    for a, b in zip(*outs):
        assert torch.equal(a, b) and torch.isfinite(a.float()).all()


@pytest.mark.parametrize("B,T,H,Hkv,dh", [(2, 300, 4, 2, 64), (1, 260, 2, 1, 128)])
def test_attention_backward_non_causal(B, T, H, Hkv, dh):
    """causal=0: every kept query attends to every kept key of its sequence
    (the lse comes from a non-causal dense forward)."""
    q, k, v, dO, lse, keep, scale = _case(B, T, H, Hkv, dh, 0.4, "gumbel", seed=5 + T, qk_std=1.2, causal=False)
    M = B * T
    idx, cu, nk = gu.compact(keep)
    Qd, Kd, Vd, dOd = (gu.bf16(a.reshape(M, -1)) for a in (q, k, v, dO))
    dQ = torch.full((M, H * dh), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    dK = torch.full((M, Hkv * dh), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    dV = torch.full((M, Hkv * dh), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    ws = torch.empty(cl.collider_attn_workspace_size(B, T, H, Hkv, dh), dtype=torch.uint8, device=gu.DEV)
    cl.collider_attn_bwd(B, T, H, Hkv, dh, 0, scale, dh, 10000.0, Qd, Kd, Vd, None, dOd, H * dh, Hkv * dh,
                         H * dh, cl.ROWS_FULL, gu.f32(lse), idx, cu, nk, dQ, dK, dV, cl.ROWS_FULL, ws)
    cl.collider_check()
    rq, rk, rv = filtered_attention_backward(q, k, v, dO, lse, keep, scale, causal=False)
    pos = np.tile(np.arange(T), B)
    rq = ops.rope_backward(rq, pos, dh, 10000.0)
    rk = ops.rope_backward(rk, pos, dh, 10000.0)
    for got, ref, nh in ((dQ, rq, H), (dK, rk, Hkv), (dV, rv, Hkv)):
        g = gu.host(got).reshape(M, nh, dh)
        assert np.all(g[keep.reshape(-1) == 0] == 0)
        assert gu.rel_err(g, ref) <= 2e-2


@pytest.mark.parametrize("B,T,H,Hkv,dh", [(2, 1100, 8, 2, 64), (1, 1300, 6, 2, 128), (1, 900, 4, 4, 64)])
def test_attention_backward_is_reproducible(B, T, H, Hkv, dh):
    """dQ sums one tile per key block: the tiles are added in key-block order,
    so dQ, dK and dV are bit-identical from run to run, on sequences of many
    key and query blocks (and still match the oracle)."""
    q, k, v, dO, lse, keep, scale = _case(B, T, H, Hkv, dh, 0.3, "gumbel", seed=17 + T, qk_std=1.5)
    M = B * T
    idx, cu, nk = gu.compact(keep)
    Qd, Kd, Vd, dOd = (gu.bf16(a.reshape(M, -1)) for a in (q, k, v, dO))
    ws = torch.empty(cl.collider_attn_workspace_size(B, T, H, Hkv, dh), dtype=torch.uint8, device=gu.DEV)
    runs = []
    for _ in range(3):
        out = [torch.full((M, n * dh), float("nan"), dtype=torch.bfloat16, device=gu.DEV) for n in (H, Hkv, Hkv)]
        cl.collider_attn_bwd(B, T, H, Hkv, dh, 1, scale, dh, 10000.0, Qd, Kd, Vd, None, dOd, H * dh, Hkv * dh,
                             H * dh, cl.ROWS_FULL, gu.f32(lse), idx, cu, nk, *out, cl.ROWS_FULL, ws)
        cl.collider_check()
        runs.append([o.clone() for o in out])
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    rq, rk, rv = filtered_attention_backward(q, k, v, dO, lse, keep, scale)
    pos = np.tile(np.arange(T), B)
    rq = ops.rope_backward(rq, pos, dh, 10000.0)
    rk = ops.rope_backward(rk, pos, dh, 10000.0)
    for got, ref, nh in zip(runs[0], (rq, rk, rv), (H, Hkv, Hkv)):
        assert gu.rel_err(gu.host(got).reshape(M, nh, dh), ref) <= 2e-2
