"""GPU parity: whole decoder block (Llama/TinyLlama-style, Qwen-style with QKV
bias and head dim 128, Phi-style parallel block) and a small stack, against
the fp64 oracle's masked full-size backward."""
import numpy as np
import pytest
import torch

import workloads
from oracle import block as ob
from oracle import stack as ost

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
cl = gu.cl

SMALL = {
    "llama": workloads.LayerShape(seed_base=81000, arch="llama", B=2, T=160, D=256, H=4, Hkv=2, dh=64, F=384,
                                  rotary_dim=64, rope_base=10000.0, norm="rms", eps=1e-5, act="swiglu",
                                  qkv_bias=False, out_bias=False, mlp_bias=False, f=0.4, mask="gumbel"),
    "qwen": workloads.LayerShape(seed_base=82000, arch="llama", B=2, T=200, D=256, H=2, Hkv=1, dh=128, F=320,
                                 rotary_dim=128, rope_base=1e6, norm="rms", eps=1e-6, act="swiglu",
                                 qkv_bias=True, out_bias=False, mlp_bias=False, f=0.4, mask="gumbel"),
    "phi": workloads.LayerShape(seed_base=83000, arch="phi", B=2, T=150, D=256, H=4, Hkv=4, dh=64, F=512,
                                rotary_dim=32, rope_base=10000.0, norm="ln", eps=1e-5, act="gelu",
                                qkv_bias=True, out_bias=True, mlp_bias=True, f=0.4, mask="span"),
}


def _oracle_case(s, f=None):
    s = s if f is None else s.with_(f=f)
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    _, saved = ob.block_forward(t["x"], w, s, round_saved=True)
    ref = ob.block_backward(t["dout"], saved, w, s, t["keep"])
    return s, w, t, saved, ref


def _compare(got, ref, keep):
    km = keep.reshape(-1) != 0
    assert np.all(got["dx"][~km] == 0)
    for k in ref:
        assert gu.rel_err(got[k], ref[k]) <= 2e-2, (k, gu.rel_err(got[k], ref[k]))


@pytest.mark.parametrize("arch", ["llama", "qwen", "phi"])
@pytest.mark.parametrize("rows", ["full", "compact"])
def test_block_backward(arch, rows):
    s, w, t, saved, ref = _oracle_case(SMALL[arch])
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    kept = np.flatnonzero(t["keep"].reshape(-1))
    n = kept.size
    if rows == "full":
        L.run(gu.bf16(t["dout"]), idx, cu, nk)
        got = L.results()
    else:
        dc = np.zeros_like(t["dout"])
        dc[:n] = t["dout"][kept]
        L.run(gu.bf16(dc), idx, cu, nk, cl.ROWS_COMPACT, cl.ROWS_COMPACT)
        got = L.results()
        dx = np.zeros_like(got["dx"])
        dx[kept] = got["dx"][:n]
        got["dx"] = dx
    cl.collider_check()
    assert set(got) == set(ref)
    _compare(got, ref, t["keep"])


@pytest.mark.parametrize("f", [0.0, 0.2, 0.6, 1.0])
def test_phi_ratio_sweep_and_degenerate(f):
    s, w, t, saved, ref = _oracle_case(SMALL["phi"], f=f)
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    got = L.results()
    cl.collider_check()
    if f == 1.0:
        for k in got:
            assert np.all(got[k] == 0), k
    else:
        _compare(got, ref, t["keep"])


def test_block_nan_poison_and_determinism():
    s, w, t, saved, ref = _oracle_case(SMALL["llama"])
    keep = t["keep"]
    km = keep.reshape(-1) == 0
    idx, cu, nk = gu.compact(keep)
    L = gu.DeviceLayer(s, w, saved)
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    a = L.results()
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    a2 = L.results()
    bad = {}
    for k, v in saved.items():
        v = np.array(v, dtype=np.float64)
        if k == "lse":
            v[np.broadcast_to((keep == 0)[:, None, :], v.shape)] = np.inf
        else:
            v[km] = np.nan
        bad[k] = v
    d2 = np.array(t["dout"])
    d2[km] = np.nan
    Lb = gu.DeviceLayer(s, w, bad)
    Lb.run(gu.bf16(d2), idx, cu, nk)
    b = Lb.results()
    cl.collider_check()
    # NaN / Inf in filtered rows reaches no output: every output of the
    # poisoned run matches the oracle (which saw the clean inputs) and is
    # bit-identical to the clean run, filtered rows of dx included
    assert set(b) == set(ref) == set(a)
    for k in ref:
        assert gu.rel_err(b[k], ref[k]) <= 2e-2, (k, gu.rel_err(b[k], ref[k]))
        assert np.array_equal(a[k], a2[k]), k
        assert np.array_equal(a[k], b[k]), k
    assert np.all(b["dx"][km] == 0)


def test_small_stack():
    ls = SMALL["llama"].with_(B=1, T=192)
    st = workloads.StackShape(seed_base=84000, layer=ls, L=2, V=512)
    t = workloads.stack_tensors(st)
    z, saved = ost.stack_forward(t["ids"], t["E"], t["layers"], t["normf_w"], t["w_lm"], ls, round_saved=True)
    ref = ost.stack_backward(z, t["targets"], t["ids"], saved, t["layers"], t["normf_w"], t["w_lm"], ls, st.V,
                             t["keep"])
    layers = [gu.DeviceLayer(ls, t["layers"][l], saved["blocks"][l]) for l in range(st.L)]
    W = (cl.LayerWeights * st.L)(*[L.weights for L in layers])
    S = (cl.LayerSaved * st.L)(*[L.saved for L in layers])
    G = (cl.LayerGrads * st.L)(*[L.grads for L in layers])
    idx, cu, nk = gu.compact(t["keep"])
    D, V, M = ls.D, st.V, ls.M
    dnf = torch.full((D,), float("nan"), device=gu.DEV)
    dlm = torch.full((D, V), float("nan"), device=gu.DEV)
    dE = torch.full((V, D), float("nan"), device=gu.DEV)
    desc = gu.layer_desc(ls)
    ws = torch.empty(cl.collider_stack_workspace_size(desc, st.L, V), dtype=torch.uint8, device=gu.DEV)
    keep_alive = [gu.bf16(z), gu.i32(t["targets"]), gu.i32(t["ids"]), gu.bf16(saved["y"]), gu.bf16(saved["xL"]),
                  gu.f32(saved["rstdf"]), gu.bf16(t["normf_w"]), gu.bf16(t["w_lm"])]
    cl.collider_stack_bwd(desc, st.L, V, W, S, *keep_alive, idx, cu, nk, G, dnf, dlm, dE, ws)
    cl.collider_check()
    assert gu.rel_err(gu.host(dlm), ref["dw_lm"]) <= 2e-2
    assert gu.rel_err(gu.host(dnf), ref["dnormf_w"]) <= 2e-2
    assert gu.rel_err(gu.host(dE), ref["dE"]) <= 2e-2
    for l in range(st.L):
        got = layers[l].results()
        for k, v in ref["blocks"][l].items():
            if k == "dx":
                continue
            assert gu.rel_err(got[k], v) <= 2e-2, (l, k, gu.rel_err(got[k], v))


def test_loss_only_filtering_baseline():
    """The prior art Collider improves on (Fig. 2b / Fig. 3): only the loss of
    filtered tokens is dropped.  On the library that is the dense backward (an
    all-kept mask) of the masked upstream gradient; it must match the oracle's
    loss-only backward, and gradients then do reach filtered rows."""
    s = SMALL["llama"]
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    keep = t["keep"]
    km = keep.reshape(-1) != 0
    _, saved = ob.block_forward(t["x"], w, s, round_saved=True)
    dmask = np.where(km[:, None], t["dout"], 0.0)
    ref = ob.block_backward(dmask, saved, w, s, keep, filter_activations=False)
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(np.ones_like(keep))
    L.run(gu.bf16(dmask), idx, cu, nk)
    got = L.results()
    cl.collider_check()
    for k in ref:
        assert gu.rel_err(got[k], ref[k]) <= 2e-2, k
    assert np.abs(got["dx"][~km]).max() > 0
