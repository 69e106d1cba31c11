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


@pytest.mark.parametrize("arch", ["llama", "qwen"])
def test_block_backward_several_query_blocks(arch):
    """Sequences of several 128-row query and key blocks (the attention's
    causal mask then falls inside blocks as well as on whole blocks), element
    by element against the oracle."""
    s, w, t, saved, ref = _oracle_case(SMALL[arch].with_(B=2, T=768))
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    got = L.results()
    cl.collider_check()
    _compare(got, ref, t["keep"])


@pytest.mark.parametrize("arch", ["llama", "qwen"])
def test_block_backward_without_a_b_s(arch):
    """A saved set without a, b and s: the backward recomputes them for the
    kept rows (from x, h and up); element by element against the oracle, on
    sequences of several query and key blocks."""
    s, w, t, saved, ref = _oracle_case(SMALL[arch].with_(B=2, T=512))
    L = gu.DeviceLayer(s, w, saved)
    L.saved.a = L.saved.b = L.saved.s = None
    idx, cu, nk = gu.compact(t["keep"])
    L.run(gu.bf16(t["dout"]), idx, cu, nk)
    got = L.results()
    cl.collider_check()
    _compare(got, ref, t["keep"])


def test_block_backward_reads_pinned_host_inputs():
    """The filtered call reads dOut and the saved set only at the kept rows,
    so they may stay in pinned host memory the device addresses directly: the
    outputs are bit-identical to those from device copies.  The dense call
    (whole tensors to TMA) and pageable host memory are refused before any
    launch, with the outputs untouched."""
    s, w, t, saved, ref = _oracle_case(SMALL["llama"].with_(B=2, T=512))
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    dout = gu.bf16(t["dout"])
    L.run(dout, idx, cu, nk)
    a = L.results()
    _compare(a, ref, t["keep"])
    by_ptr = {x.data_ptr(): x for x in L.keep_alive}
    fields = [f for f, _ in cl.LayerSaved._fields_]
    pinned = {f: by_ptr[getattr(L.saved, f)].cpu().pin_memory() for f in fields if getattr(L.saved, f)}
    hs = cl.LayerSaved(**{f: v.data_ptr() for f, v in pinned.items()})
    hdout = dout.cpu().pin_memory()
    for v in L.grads_t.values():
        v.fill_(float("nan"))
    L.dx.fill_(float("nan"))
    cl.collider_layer_bwd(L.desc, L.weights, hs, hdout, cl.ROWS_FULL, idx, cu, nk, L.grads, cl.ROWS_FULL, L.ws)
    b = L.results()
    cl.collider_check()
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    for v in L.grads_t.values():
        v.fill_(7.0)
    with pytest.raises(cl.ColliderError):
        cl.collider_layer_bwd(L.desc, L.weights, hs, hdout, cl.ROWS_FULL, None, None, None, L.grads, cl.ROWS_FULL,
                              L.ws)
    with pytest.raises(cl.ColliderError):
        cl.collider_layer_bwd(L.desc, L.weights, L.saved, dout.cpu(), cl.ROWS_FULL, idx, cu, nk, L.grads,
                              cl.ROWS_FULL, L.ws)
    torch.cuda.synchronize()
    for v in L.grads_t.values():
        assert torch.all(v == 7.0)


def test_block_backward_is_reproducible():
    """Every output of the block -- dx and the weight gradients below the
    attention (dw_qkv, dnorm1_w) included -- is bit-identical run to run, on
    sequences of several key blocks, because every reduction has a fixed order."""
    s = SMALL["llama"].with_(B=2, T=1100)
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    _, saved = ob.block_forward(t["x"], w, s, round_saved=True)
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    outs = []
    for _ in range(3):
        L.run(gu.bf16(t["dout"]), idx, cu, nk)
        outs.append(L.results())
        cl.collider_check()
    for o in outs[1:]:
        for k in outs[0]:
            assert np.array_equal(outs[0][k], o[k]), k


@pytest.mark.parametrize("arch", ["llama", "qwen", "phi"])
def test_dense_call_is_the_all_kept_backward(arch):
    """idx, cu_kept, n_kept all NULL: the unfiltered dense backward reads FULL
    rows in place (no gather, no scatter).  It matches the oracle with nothing
    filtered and is bit-identical to the filtered path run on an all-kept
    mask (M = 320 or 400 or 300 rows: not whole 128-row tiles)."""
    s = SMALL[arch].with_(f=0.0)
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    keep = np.ones((s.B, s.T), dtype=np.uint8)
    _, saved = ob.block_forward(t["x"], w, s, round_saved=True)
    ref = ob.block_backward(t["dout"], saved, w, s, keep)
    L = gu.DeviceLayer(s, w, saved)
    dout = gu.bf16(t["dout"])
    L.run(dout, None, None, None)
    dense = L.results()
    cl.collider_check()
    idx, cu, nk = gu.compact(keep)
    L.run(dout, idx, cu, nk)
    masked = L.results()
    cl.collider_check()
    for k in ref:
        assert gu.rel_err(dense[k], ref[k]) <= 2e-2, (k, gu.rel_err(dense[k], ref[k]))
        assert np.array_equal(dense[k], masked[k]), k


def test_dense_call_rejects_a_partial_index():
    s = SMALL["llama"]
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    _, saved = ob.block_forward(t["x"], w, s, round_saved=True)
    L = gu.DeviceLayer(s, w, saved)
    idx, cu, nk = gu.compact(t["keep"])
    with pytest.raises(cl.ColliderError, match="idx/cu_kept/n_kept"):
        L.run(gu.bf16(t["dout"]), idx, None, None)


@pytest.mark.parametrize("lean", [False, True])
def test_small_stack(lean):
    """A two-block stack against the oracle's stack backward; lean: every
    block's saved set without a, b and s (recomputed for the kept rows)."""
    ls = SMALL["llama"].with_(B=1, T=192)
    st = workloads.StackShape(seed_base=84000, layer=ls, L=2, V=512)
    t = workloads.stack_tensors(st)
    z, saved = ost.stack_forward(t["ids"], t["E"], t["layers"], t["normf_w"], t["w_lm"], ls, round_saved=True)
    ref = ost.stack_backward(z, t["targets"], t["ids"], saved, t["layers"], t["normf_w"], t["w_lm"], ls, st.V,
                             t["keep"])
    layers = [gu.DeviceLayer(ls, t["layers"][l], saved["blocks"][l]) for l in range(st.L)]
    if lean:
        for L in layers:
            L.saved.a = L.saved.b = L.saved.s = None
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


def test_small_stack_dense_call():
    """The stack's dense call (NULL index) is bit-identical to its filtered path
    on an all-kept mask, and matches the oracle with nothing filtered."""
    ls = SMALL["llama"].with_(B=1, T=192, f=0.0)
    st = workloads.StackShape(seed_base=85000, layer=ls, L=2, V=512)
    t = workloads.stack_tensors(st)
    keep = np.ones((ls.B, ls.T), dtype=np.uint8)
    z, saved = ost.stack_forward(t["ids"], t["E"], t["layers"], t["normf_w"], t["w_lm"], ls, round_saved=True)
    ref = ost.stack_backward(z, t["targets"], t["ids"], saved, t["layers"], t["normf_w"], t["w_lm"], ls, st.V, keep)
    layers = [gu.DeviceLayer(ls, t["layers"][l], saved["blocks"][l]) for l in range(st.L)]
    W = (cl.LayerWeights * st.L)(*[L.weights for L in layers])
    S = (cl.LayerSaved * st.L)(*[L.saved for L in layers])
    G = (cl.LayerGrads * st.L)(*[L.grads for L in layers])
    D, V = ls.D, st.V
    desc = gu.layer_desc(ls)
    ws = torch.empty(cl.collider_stack_workspace_size(desc, st.L, V), dtype=torch.uint8, device=gu.DEV)
    ins = [gu.bf16(z), gu.i32(t["targets"]), gu.i32(t["ids"]), gu.bf16(saved["y"]), gu.bf16(saved["xL"]),
           gu.f32(saved["rstdf"]), gu.bf16(t["normf_w"]), gu.bf16(t["w_lm"])]
    res = []
    for index in ((None, None, None), gu.compact(keep)):
        outs = [torch.full(shp, float("nan"), device=gu.DEV) for shp in ((D,), (D, V), (V, D))]
        cl.collider_stack_bwd(desc, st.L, V, W, S, *ins, *index, G, *outs, ws)
        cl.collider_check()
        res.append([gu.host(o) for o in outs] + [layers[l].results() for l in range(st.L)])
    (dnf, dlm, dE), (dnf2, dlm2, dE2) = res[0][:3], res[1][:3]
    assert np.array_equal(dnf, dnf2) and np.array_equal(dlm, dlm2) and np.array_equal(dE, dE2)
    assert gu.rel_err(dlm, ref["dw_lm"]) <= 2e-2 and gu.rel_err(dE, ref["dE"]) <= 2e-2
    for l in range(st.L):
        a, b = res[0][3 + l], res[1][3 + l]
        for k, v in ref["blocks"][l].items():
            if k == "dx":
                continue
            assert np.array_equal(a[k], b[k]), (l, k)
            assert gu.rel_err(a[k], v) <= 2e-2, (l, k)
