"""Helpers for the GPU parity tests: upload oracle inputs, call libcollider
through its C ABI, bring results back as float64 numpy arrays."""
from __future__ import annotations

import math

import numpy as np
import torch

import sparse_backward_gemm_gb300 as cl

DEV = "cuda:0"


def bf16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32))).to(DEV).to(torch.bfloat16)


def f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32))).to(DEV)


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    m = np.max(np.abs(ref)) if ref.size else 0.0
    if m == 0.0:
        return 0.0 if np.all(got == 0) else math.inf
    return float(np.max(np.abs(got - ref)) / m)


def compact(keep: np.ndarray):
    """Run collider_compact on the GPU; returns (idx, cu_kept, n_kept) tensors."""
    B, T = keep.shape
    mask = torch.from_numpy(np.ascontiguousarray(keep.astype(np.uint8))).to(DEV)
    idx = torch.full((B * T,), -1, dtype=torch.int32, device=DEV)
    cu = torch.full((B + 1,), -1, dtype=torch.int32, device=DEV)
    nk = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    wsb = cl.collider_compact_workspace_size(B, T)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=DEV) if wsb else None
    cl.collider_compact(mask, B, T, idx, cu, nk, ws)
    return idx, cu, nk


def layer_desc(s) -> cl.LayerDesc:
    return cl.LayerDesc(arch=cl.ARCH_LLAMA if s.arch == "llama" else cl.ARCH_PHI, B=s.B, T=s.T, D=s.D, H=s.H,
                        Hkv=s.Hkv, dh=s.dh, F=s.F, rotary_dim=s.rotary_dim, rope_base=s.rope_base,
                        norm=cl.NORM_RMS if s.norm == "rms" else cl.NORM_LAYER, eps=s.eps,
                        act=cl.ACT_SWIGLU if s.act == "swiglu" else cl.ACT_GELU_TANH, qkv_bias=int(s.qkv_bias),
                        out_bias=int(s.out_bias), mlp_bias=int(s.mlp_bias))


class DeviceLayer:
    """A block's weights, saved set and gradient buffers on the device."""

    def __init__(self, s, w: dict, saved: dict):
        self.s = s
        self.keep_alive = []
        g = lambda k: self._t(bf16(w[k])) if k in w else None
        self.weights = cl.LayerWeights(norm1_w=g("norm1_w"), w_qkv=g("w_qkv"), w_o=g("w_o"),
                                       norm2_w=g("norm2_w"), w_up=g("w_up"), w_down=g("w_down"))
        sb = lambda k: self._t(bf16(saved[k])) if k in saved else None
        sf = lambda k: self._t(f32(saved[k])) if k in saved else None
        up = saved["gu"] if s.arch == "llama" else saved["f1"]
        self.saved = cl.LayerSaved(x=sb("x"), a=sb("a"), mean1=sf("mean1"), rstd1=sf("rstd1"), qkv=sb("qkv"),
                                   o=sb("o"), lse=sf("lse"), h=sb("h"), b=sb("b"), rstd2=sf("rstd2"),
                                   up=self._t(bf16(up)), s=sb("s"))
        self.grads_t = {}
        shapes = dict(dnorm1_w=(s.D,), dw_qkv=(s.D, s.Nqkv), dw_o=(s.H * s.dh, s.D), dw_up=(s.D, s.Nup),
                      dw_down=(s.F, s.D))
        if s.norm == "ln":
            shapes["dnorm1_b"] = (s.D,)
        if s.arch == "llama":
            shapes["dnorm2_w"] = (s.D,)
        if s.qkv_bias:
            shapes["db_qkv"] = (s.Nqkv,)
        if s.out_bias:
            shapes["db_o"] = (s.D,)
        if s.mlp_bias:
            shapes["db_up"] = (s.Nup,)
            shapes["db_down"] = (s.D,)
        for k, shp in shapes.items():
            self.grads_t[k] = torch.full(shp, float("nan"), dtype=torch.float32, device=DEV)
        self.dx = torch.full((s.M, s.D), float("nan"), dtype=torch.bfloat16, device=DEV)
        self.grads = cl.LayerGrads(dx=self.dx.data_ptr(), **{k: v.data_ptr() for k, v in self.grads_t.items()})
        self.desc = layer_desc(s)
        self.ws = torch.empty(cl.collider_layer_workspace_size(self.desc), dtype=torch.uint8, device=DEV)

    def _t(self, t):
        self.keep_alive.append(t)
        return t.data_ptr()

    def run(self, dout_t, idx, cu, nk, dout_rows=cl.ROWS_FULL, dx_rows=cl.ROWS_FULL):
        cl.collider_layer_bwd(self.desc, self.weights, self.saved, dout_t, dout_rows, idx, cu, nk, self.grads,
                              dx_rows, self.ws)

    def results(self) -> dict:
        torch.cuda.synchronize()
        out = {k: host(v) for k, v in self.grads_t.items()}
        out["dx"] = host(self.dx)
        return out
