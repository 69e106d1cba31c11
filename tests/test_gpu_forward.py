"""GPU parity: the dense forward of one block (collider_layer_fwd) against the
fp64 oracle's forward, which rounds each saved tensor to its storage type.

Small shapes (Llama-, Qwen- and Phi-style, ragged sequence lengths) are
compared element by element; the full-size blocks are compared on one whole
sequence (sequences are independent in the forward), the last one of the
batch so the sequence offset is exercised.  The saved set the GPU forward
writes is also fed to the GPU backward and checked against the oracle's
backward, so the two halves agree on every layout."""
import numpy as np
import pytest
import torch

import workloads
from oracle import block as ob

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
cl = gu.cl

BF16_TOL = 2e-2     # bf16 outputs: max|err| / max|ref|
STAT_TOL = 1e-3     # f32 row statistics (lse, mean, rstd) computed from bf16 operands

SMALL = {
    "llama": workloads.LayerShape(seed_base=91000, arch="llama", B=2, T=160, D=256, H=4, Hkv=2, dh=64, F=384,
                                  rotary_dim=64, rope_base=10000.0, norm="rms", eps=1e-5, act="swiglu",
                                  qkv_bias=False, out_bias=False, mlp_bias=False, f=0.4, mask="gumbel"),
    "gqa4": workloads.LayerShape(seed_base=91500, arch="llama", B=3, T=300, D=256, H=8, Hkv=2, dh=64, F=256,
                                 rotary_dim=64, rope_base=10000.0, norm="rms", eps=1e-5, act="swiglu",
                                 qkv_bias=False, out_bias=False, mlp_bias=False, f=0.4, mask="gumbel"),
    "qwen": workloads.LayerShape(seed_base=92000, arch="llama", B=2, T=200, D=256, H=2, Hkv=1, dh=128, F=320,
                                 rotary_dim=128, rope_base=1e6, norm="rms", eps=1e-6, act="swiglu",
                                 qkv_bias=True, out_bias=False, mlp_bias=False, f=0.4, mask="gumbel"),
    "phi": workloads.LayerShape(seed_base=93000, arch="phi", B=2, T=150, D=256, H=4, Hkv=4, dh=64, F=512,
                                rotary_dim=32, rope_base=10000.0, norm="ln", eps=1e-5, act="gelu",
                                qkv_bias=True, out_bias=True, mlp_bias=True, f=0.4, mask="span"),
}


class DeviceForward:
    """A block's parameters and the buffers the forward writes, on the device."""

    def __init__(self, s, w: dict):
        self.s = s
        self.keep = []
        g = lambda k: self._p(gu.bf16(w[k])) if k in w else None
        self.params = cl.LayerParams(norm1_w=g("norm1_w"), norm1_b=g("norm1_b"), w_qkv=g("w_qkv"),
                                     b_qkv=g("b_qkv"), w_o=g("w_o"), b_o=g("b_o"), norm2_w=g("norm2_w"),
                                     w_up=g("w_up"), b_up=g("b_up"), w_down=g("w_down"), b_down=g("b_down"))
        M = s.M
        nan = float("nan")
        bf = lambda *shp: torch.full(shp, nan, dtype=torch.bfloat16, device=gu.DEV)
        f32 = lambda *shp: torch.full(shp, nan, dtype=torch.float32, device=gu.DEV)
        self.t = dict(a=bf(M, s.D), rstd1=f32(M), qkv=bf(M, s.Nqkv), o=bf(M, s.H * s.dh), lse=f32(s.B, s.H, s.T),
                      up=bf(M, s.Nup))
        if s.arch == "llama":
            self.t.update(h=bf(M, s.D), b=bf(M, s.D), rstd2=f32(M), s=bf(M, s.F))
        else:
            self.t["mean1"] = f32(M)
        self.acts = cl.LayerActs(**{k: v.data_ptr() for k, v in self.t.items()})
        self.y = bf(M, s.D)
        self.desc = gu.layer_desc(s)
        self.ws = torch.empty(cl.collider_layer_fwd_workspace_size(self.desc), dtype=torch.uint8, device=gu.DEV)

    def _p(self, t):
        self.keep.append(t)
        return t.data_ptr()

    def run(self, x_t):
        cl.collider_layer_fwd(self.desc, self.params, x_t, self.y, self.acts, self.ws)

    def results(self) -> dict:
        torch.cuda.synchronize()
        out = {k: gu.host(v) for k, v in self.t.items()}
        out["y"] = gu.host(self.y)
        return out

    def saved_struct(self, x_t) -> "cl.LayerSaved":
        p = lambda k: self.t[k].data_ptr() if k in self.t else None
        return cl.LayerSaved(x=x_t.data_ptr(), a=p("a"), mean1=p("mean1"), rstd1=p("rstd1"), qkv=p("qkv"), o=p("o"),
                             lse=p("lse"), h=p("h"), b=p("b"), rstd2=p("rstd2"), up=p("up"), s=p("s"))


def _oracle_names(s):
    """GPU saved-set name -> oracle saved-set name."""
    m = dict(a="a", rstd1="rstd1", qkv="qkv", o="o", lse="lse", up="gu" if s.arch == "llama" else "f1")
    if s.arch == "llama":
        m.update(h="h", b="b", rstd2="rstd2", s="s")
    else:
        m["mean1"] = "mean1"
    return m


def _compare(s, got, out_ref, sv_ref, rows=slice(None), lse_b=slice(None)):
    for k, ko in _oracle_names(s).items():
        ref = sv_ref[ko]
        g = got[k][lse_b] if k == "lse" else got[k][rows]
        tol = STAT_TOL if k in ("lse", "mean1", "rstd1", "rstd2") else BF16_TOL
        err = gu.rel_err(g.reshape(ref.shape), ref)
        assert err <= tol, (k, err)
    err = gu.rel_err(got["y"][rows], out_ref)
    assert err <= BF16_TOL, ("y", err)


@pytest.mark.parametrize("arch", list(SMALL))
def test_block_forward(arch):
    s = SMALL[arch]
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    out_ref, sv_ref = ob.block_forward(t["x"], w, s, round_saved=True)
    F = DeviceForward(s, w)
    x_t = gu.bf16(t["x"])
    F.run(x_t)
    got = F.results()
    cl.collider_check()
    _compare(s, got, out_ref, sv_ref)
    # no atomics anywhere in the forward: a second run is bit-identical
    F.run(x_t)
    again = F.results()
    for k in got:
        assert np.array_equal(got[k], again[k]), k


@pytest.mark.parametrize("arch", ["llama", "qwen", "phi"])
def test_forward_feeds_backward(arch):
    """The GPU forward's saved set drives the GPU backward to the oracle's gradients."""
    s = SMALL[arch]
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    _, sv_ref = ob.block_forward(t["x"], w, s, round_saved=True)
    ref = ob.block_backward(t["dout"], sv_ref, w, s, t["keep"])
    F = DeviceForward(s, w)
    x_t = gu.bf16(t["x"])
    F.run(x_t)
    L = gu.DeviceLayer(s, w, sv_ref)          # weights and gradient buffers; saved set replaced below
    L.saved = F.saved_struct(x_t)
    idx, cu, nk = gu.compact(t["keep"])
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    got = L.results()
    cl.collider_check()
    km = t["keep"].reshape(-1) != 0
    assert np.all(got["dx"][~km] == 0)
    for k in ref:
        assert gu.rel_err(got[k], ref[k]) <= BF16_TOL, (k, gu.rel_err(got[k], ref[k]))


@pytest.mark.parametrize("arch", ["llama", "qwen"])
def test_backward_recomputes_a_b_s_exactly(arch):
    """A filtered backward given a saved set without a, b and s recomputes them
    for the kept rows with the forward's roundings: every gradient is
    bit-identical to the one from the forward's own a, b and s.  The dense
    call, which reads them in place, refuses such a saved set."""
    s = SMALL[arch].with_(T=640)
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    _, sv_ref = ob.block_forward(t["x"], w, s, round_saved=True)
    ref = ob.block_backward(t["dout"], sv_ref, w, s, t["keep"])
    F = DeviceForward(s, w)
    x_t = gu.bf16(t["x"])
    F.run(x_t)
    L = gu.DeviceLayer(s, w, sv_ref)
    full = F.saved_struct(x_t)
    L.saved = full
    idx, cu, nk = gu.compact(t["keep"])
    dout = gu.bf16(t["dout"])
    L.run(dout, idx, cu, nk)
    a = L.results()
    part = cl.LayerSaved(**{f: getattr(full, f) for f, _ in cl.LayerSaved._fields_})
    part.a = part.b = part.s = None
    L.saved = part
    for v in L.grads_t.values():
        v.fill_(float("nan"))
    L.dx.fill_(float("nan"))
    L.run(dout, idx, cu, nk)
    b = L.results()
    cl.collider_check()
    for k in a:
        assert np.array_equal(a[k], b[k]), k
        assert gu.rel_err(b[k], ref[k]) <= BF16_TOL, (k, gu.rel_err(b[k], ref[k]))
    with pytest.raises(cl.ColliderError):
        L.run(dout, None, None, None)


FULL = ["tinyllama_layer", "qwen25_layer", "phi15_layer"]


@pytest.mark.parametrize("name", FULL)
def test_block_forward_full_size(name):
    """Full-size block on the GPU; the last sequence against the oracle's forward of that sequence."""
    s = workloads.WORKLOADS[name]
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    F = DeviceForward(s, w)
    F.run(gu.bf16(t["x"]))
    got = F.results()
    cl.collider_check()
    b = s.B - 1
    rows = slice(b * s.T, (b + 1) * s.T)
    s1 = s.with_(B=1)
    out_ref, sv_ref = ob.block_forward(t["x"][rows], w, s1, round_saved=True)
    _compare(s1, got, out_ref, sv_ref, rows=rows, lse_b=slice(b, b + 1))
