"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (FULL dOut rows in, FULL dx rows out, one compaction per
step).

Single blocks (TinyLlama-, Qwen2.5- and Phi-1.5-shaped) are compared with the
fp64 oracle element by element over every output tensor.  The 22-block stack
at 8192 tokens is too large for the oracle as a whole: its LM head, final norm
and last block are checked against the oracle, the rest by properties that hold
at any size (finite, filtered rows zero, reproducible weight gradients,
embedding rows only at kept token ids).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import block as ob
from oracle import ops

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

gu = pytest.importorskip("gpu_util")
cl = gu.cl


def _run_block(s):
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    _, saved = ob.block_forward(t["x"], w, s, round_saved=True)
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    got = L.results()
    cl.collider_check()
    ref = ob.block_backward(t["dout"], saved, w, s, t["keep"])
    return got, ref, t["keep"]


def _compare(got, ref, keep):
    km = keep.reshape(-1) != 0
    assert np.all(got["dx"][~km] == 0)
    worst = {k: gu.rel_err(got[k], ref[k]) for k in ref}
    assert max(worst.values()) <= 2e-2, worst


@pytest.mark.parametrize("name", ["tinyllama_layer", "qwen25_layer"])
def test_full_size_block(name):
    s = workloads.WORKLOADS[name]
    got, ref, keep = _run_block(s)
    _compare(got, ref, keep)


@pytest.mark.parametrize("f", [0.0, 0.2, 0.4, 0.6])
def test_full_size_phi_ratio_sweep(f):
    s = workloads.WORKLOADS["phi15_layer"].with_(f=f)
    got, ref, keep = _run_block(s)
    _compare(got, ref, keep)


def _gpu_stack_forward(st, t):
    """Dense bf16 stack forward with torch on the GPU (input preparation)."""
    from torch_forward import gpu_forward
    ls = st.layer
    dev = torch.device(gu.DEV)
    E = torch.from_numpy(t["E"]).to(dev).bfloat16()
    ids = torch.from_numpy(t["ids"].astype(np.int64)).to(dev)
    x = E[ids]
    blocks, Ws = [], []
    for w in t["layers"]:
        W = {k: torch.from_numpy(v).to(dev).bfloat16() for k, v in w.items()}
        sv = gpu_forward(ls, W, x)
        blocks.append(sv)
        Ws.append(W)
        xf = sv["h"].float() + sv["s"].float() @ W["w_down"].float()
        x = xf.bfloat16()
    xf = x.float()
    rstd = torch.rsqrt(xf.pow(2).mean(-1) + ls.eps)
    nf = torch.from_numpy(t["normf_w"]).to(dev).bfloat16()
    y = (xf * rstd[:, None] * nf.float()).bfloat16()
    wlm = torch.from_numpy(t["w_lm"]).to(dev).bfloat16()
    z = (y.float() @ wlm.float()).bfloat16()
    return blocks, Ws, x, rstd, y, z, nf, wlm


def test_full_size_stack():
    st = workloads.WORKLOADS["tinyllama_stack"]
    ls = st.layer
    t = workloads.stack_tensors(st)
    with torch.no_grad():
        blocks, Ws, xL, rstdf, y, z, nf, wlm = _gpu_stack_forward(st, t)
    D, V, M, L = ls.D, st.V, ls.M, st.L
    desc = gu.layer_desc(ls)
    Wc = (cl.LayerWeights * L)(*[cl.LayerWeights(**{k: W[k].data_ptr() for k in ("norm1_w", "w_qkv", "w_o",
                                                                                  "norm2_w", "w_up", "w_down")})
                                 for W in Ws])
    Sc = (cl.LayerSaved * L)(*[cl.LayerSaved(**{k: sv[k].data_ptr() for k in sv}) for sv in blocks])
    grads = []
    for _ in range(L):
        g = {k: torch.empty(shp, dtype=torch.float32, device=gu.DEV) for k, shp in
             dict(dnorm1_w=(D,), dw_qkv=(D, ls.Nqkv), dw_o=(ls.H * ls.dh, D), dnorm2_w=(D,), dw_up=(D, ls.Nup),
                  dw_down=(ls.F, D)).items()}
        grads.append(g)
    Gc = (cl.LayerGrads * L)(*[cl.LayerGrads(dx=None, **{k: v.data_ptr() for k, v in g.items()}) for g in grads])
    idx, cu, nk = gu.compact(t["keep"])
    targets = gu.i32(t["targets"])
    ids = gu.i32(t["ids"])
    dnf = torch.empty(D, device=gu.DEV)
    dlm = torch.empty(D, V, device=gu.DEV)
    dE = torch.empty(V, D, device=gu.DEV)
    ws = torch.empty(cl.collider_stack_workspace_size(desc, L, V), dtype=torch.uint8, device=gu.DEV)

    def run():
        cl.collider_stack_bwd(desc, L, V, Wc, Sc, z, targets, ids, y, xL, rstdf, nf, wlm, idx, cu, nk, Gc, dnf,
                              dlm, dE, ws)
        cl.collider_check()
        return gu.host(dlm), gu.host(dnf), gu.host(dE), [{k: gu.host(v) for k, v in g.items()} for g in grads]

    dlm1, dnf1, dE1, g1 = run()
    dlm2, dnf2, dE2, g2 = run()
    km = t["keep"].reshape(-1) != 0
    # properties at full size
    for a in [dlm1, dnf1, dE1] + [v for g in g1 for v in g.values()]:
        assert np.all(np.isfinite(a))
    # bit-reproducible where no attention reduce-add lies upstream: the LM
    # head, the final norm and the MLP / output projection of the last block;
    # below that the f32 reduce order of dQ, dK, dV varies run to run
    assert np.array_equal(dlm1, dlm2) and np.array_equal(dnf1, dnf2)
    for k in ("dw_down", "dw_up", "dnorm2_w", "dw_o"):
        assert np.array_equal(g1[-1][k], g2[-1][k]), k
    for l, (la, lb) in enumerate(zip(g1, g2)):
        for k in la:
            e = gu.rel_err(la[k], lb[k])
            assert e <= 5e-2, (l, k, e)
    seen = set(np.flatnonzero(np.abs(dE1).sum(1)).tolist())
    assert seen <= set(t["ids"][km].tolist())

    # the oracle on the LM head, final norm and last block
    zk = gu.host(z)
    dz = ops.ce_backward(zk, t["targets"], km)
    yk = np.where(km[:, None], gu.host(y), 0.0)
    assert gu.rel_err(dlm1, yk.T @ dz) <= 2e-2
    dy = dz @ gu.host(wlm).T
    dx22, dnf_ref = ops.rmsnorm_backward(dy, np.where(km[:, None], gu.host(xL), 0.0),
                                         np.where(km, gu.host(rstdf), 0.0), gu.host(nf))
    assert gu.rel_err(dnf1, dnf_ref) <= 2e-2
    last = {k: gu.host(v) for k, v in blocks[-1].items()}
    last["gu"] = last.pop("up")       # the oracle names the saved [gate | up] projection "gu"
    wl = {k: v.astype(np.float64) for k, v in t["layers"][-1].items()}
    ref = ob.block_backward(dx22, last, wl, ls, t["keep"])
    for k in ("dw_down", "dw_up", "dnorm2_w", "dw_o", "dw_qkv", "dnorm1_w"):
        assert gu.rel_err(g1[-1][k], ref[k]) <= 2e-2, k
