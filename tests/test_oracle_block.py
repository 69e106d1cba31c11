"""Pins for oracle.block (and oracle.stack): float64 autograd of the
independently written surrogate forward, finite differences of it, and the
invariants of the filtered backward."""
import numpy as np
import pytest
import torch

from oracle import block as ob
from oracle import stack as ost
import surrogate_torch as sg
import workloads

TINY_LLAMA = workloads.LayerShape(seed_base=91000, arch="llama", B=2, T=8, D=16, H=2, Hkv=1, dh=8,
                                  F=24, rotary_dim=8, rope_base=10000.0, norm="rms", eps=1e-5,
                                  act="swiglu", qkv_bias=False, out_bias=False, mlp_bias=False,
                                  f=0.4, mask="gumbel")
TINY_QWEN = TINY_LLAMA.with_(seed_base=92000, H=4, Hkv=2, qkv_bias=True, eps=1e-6, rope_base=1e6)
TINY_PHI = workloads.LayerShape(seed_base=93000, arch="phi", B=2, T=8, D=16, H=2, Hkv=2, dh=8, F=24,
                                rotary_dim=4, rope_base=10000.0, norm="ln", eps=1e-5, act="gelu",
                                qkv_bias=True, out_bias=True, mlp_bias=True, f=0.4, mask="span")
SHAPES = [TINY_LLAMA, TINY_QWEN, TINY_PHI]


def big_weights(s, seed):
    """Weights with std 0.3 so attention is far from uniform (sharper pins)."""
    w = workloads.layer_weights(s, seed_base=seed)
    return {k: ((v.astype(np.float64) - (1.0 if k in ("norm1_w", "norm2_w") else 0.0)) * 15.0
                + (1.0 if k in ("norm1_w", "norm2_w") else 0.0)) for k, v in w.items()}


def _t(d):
    return {k: torch.tensor(np.asarray(v, dtype=np.float64), requires_grad=True) for k, v in d.items()}


def _rel(a, b):
    return np.max(np.abs(np.asarray(a) - np.asarray(b))) / max(np.max(np.abs(b)), 1e-300)


def _case(s, seed=0):
    w = big_weights(s, s.seed_base + seed)
    rng = np.random.default_rng(s.seed_base + seed)
    x = rng.normal(size=(s.M, s.D))
    dout = rng.normal(size=(s.M, s.D))
    keep = workloads.keep_mask(s.B, s.T, s.f, s.mask, seed=s.seed_base + seed)
    return w, x, dout, keep


@pytest.mark.parametrize("s", SHAPES, ids=["llama", "qwen", "phi"])
def test_block_matches_autograd_of_surrogate(s):
    w, x, dout, keep = _case(s)
    out, saved = ob.block_forward(x, w, s, round_saved=False)
    g = ob.block_backward(dout, saved, w, s, keep)
    tw = _t(w)
    tx = torch.tensor(x, requires_grad=True)
    kt = torch.tensor(keep != 0)
    tout = sg.block(tx, tw, s, keep=kt)
    assert _rel(tout.detach().numpy(), out) < 1e-12
    m = kt.reshape(-1).to(torch.float64)[:, None]
    (tout * torch.tensor(dout) * m).sum().backward()
    assert _rel(g["dx"], tx.grad.numpy()) < 1e-11
    for name, t in tw.items():
        assert _rel(g["d" + name], t.grad.numpy()) < 1e-11, name
    assert set("d" + n for n in tw) | {"dx"} == set(g)


@pytest.mark.parametrize("s", SHAPES, ids=["llama", "qwen", "phi"])
def test_block_zero_filtering_is_dense_autograd(s):
    w, x, dout, _ = _case(s, seed=1)
    keep = np.ones((s.B, s.T), np.uint8)
    _, saved = ob.block_forward(x, w, s, round_saved=False)
    g = ob.block_backward(dout, saved, w, s, keep)
    tw = _t(w)
    tx = torch.tensor(x, requires_grad=True)
    (sg.block(tx, tw, s, keep=None) * torch.tensor(dout)).sum().backward()
    assert _rel(g["dx"], tx.grad.numpy()) < 1e-11
    for name, t in tw.items():
        assert _rel(g["d" + name], t.grad.numpy()) < 1e-11, name


def test_block_finite_differences_of_surrogate():
    s = TINY_LLAMA
    w, x, dout, keep = _case(s, seed=2)
    _, saved = ob.block_forward(x, w, s, round_saved=False)
    g = ob.block_backward(dout, saved, w, s, keep)
    kt = torch.tensor(keep != 0)
    m = kt.reshape(-1).to(torch.float64)[:, None]
    frozen = {}
    tw0 = {k: torch.tensor(v) for k, v in w.items()}
    sg.block(torch.tensor(x), tw0, s, keep=kt, frozen=frozen)

    def L(xx, ww):
        return float((sg.block(torch.tensor(xx), {k: torch.tensor(v) for k, v in ww.items()}, s,
                               keep=kt, frozen=frozen) * torch.tensor(dout) * m).sum())
    h = 1e-6
    rng = np.random.default_rng(3)
    for _ in range(12):
        c = (int(rng.integers(0, s.M)), int(rng.integers(0, s.D)))
        xp, xm = x.copy(), x.copy()
        xp[c] += h; xm[c] -= h
        fd = (L(xp, w) - L(xm, w)) / (2 * h)
        assert abs(fd - g["dx"][c]) < 2e-6 * max(1, np.abs(g["dx"]).max())
    for name in ("w_qkv", "w_o", "w_up", "w_down", "norm1_w", "norm2_w"):
        for _ in range(4):
            c = tuple(int(rng.integers(0, n)) for n in w[name].shape)
            wp = dict(w); wm = dict(w)
            wp[name] = w[name].copy(); wp[name][c] += h
            wm[name] = w[name].copy(); wm[name][c] -= h
            fd = (L(x, wp) - L(x, wm)) / (2 * h)
            assert abs(fd - g["d" + name][c]) < 2e-6 * max(1, np.abs(g["d" + name]).max()), name


SAVED_ROWS = ("x", "a", "rstd1", "mean1", "qkv", "o", "h", "b", "rstd2", "gu", "s", "f1")


@pytest.mark.parametrize("s", SHAPES, ids=["llama", "qwen", "phi"])
def test_block_invariants(s):
    w, x, dout, keep = _case(s, seed=4)
    _, saved = ob.block_forward(x, w, s, round_saved=True)
    g = ob.block_backward(dout, saved, w, s, keep)
    km = keep.reshape(-1) != 0
    assert np.all(g["dx"][~km] == 0)
    # filtered rows of every saved tensor and of dOut replaced with junk
    # (lse of filtered query positions too): every gradient is unchanged
    rng = np.random.default_rng(5)
    bad = dict(saved)
    for k in SAVED_ROWS:
        if k in bad:
            t = np.array(bad[k], dtype=np.float64)
            t[~km] = rng.normal(size=t[~km].shape) * 1e6
            t[np.flatnonzero(~km)[:1]] = np.nan
            bad[k] = t
    lse = np.array(saved["lse"])
    lse[np.broadcast_to((keep == 0)[:, None, :], lse.shape)] = np.inf
    bad["lse"] = lse
    d2 = np.array(dout)
    d2[~km] = np.nan
    g2 = ob.block_backward(d2, bad, w, s, keep)
    for k in g:
        assert np.array_equal(g[k], g2[k]), k
    # and permuting the filtered rows among themselves changes nothing either
    perm = np.flatnonzero(~km)
    p2 = dict(saved)
    for k in SAVED_ROWS:
        if k in p2:
            t = np.array(p2[k]); t[perm] = t[perm[::-1]]; p2[k] = t
    g3 = ob.block_backward(dout, p2, w, s, keep)
    for k in g:
        assert np.array_equal(g[k], g3[k]), k
    # 100% filtered: all zero
    g0 = ob.block_backward(dout, saved, w, s, np.zeros_like(keep))
    for k in g0:
        assert np.all(g0[k] == 0), k


def test_loss_only_filtering_spreads_density():
    """Fig. 3: with only the loss filtered, gradients reach filtered tokens'
    rows (G_V is dense and density passes to earlier layers)."""
    s = TINY_LLAMA
    w, x, dout, keep = _case(s, seed=6)
    km = keep.reshape(-1) != 0
    _, saved = ob.block_forward(x, w, s, round_saved=False)
    dmask = np.where(km[:, None], dout, 0.0)
    g = ob.block_backward(dmask, saved, w, s, keep)
    ga = ob.block_backward(dmask, saved, w, s, keep, filter_activations=False)
    assert np.all(g["dx"][~km] == 0)
    assert np.all(np.abs(ga["dx"][~km]).max(axis=1) > 0)
    # the MLP half sees only kept rows in both (token-wise, dOut rows zero)
    for k in ("dw_down", "dw_up", "dnorm2_w"):
        np.testing.assert_allclose(g[k], ga[k], rtol=1e-12, atol=1e-12)
    assert not np.allclose(g["dw_qkv"], ga["dw_qkv"])
    # and with nothing filtered the two agree
    ones = np.ones_like(keep)
    g1 = ob.block_backward(dout, saved, w, s, ones)
    g2 = ob.block_backward(dout, saved, w, s, ones, filter_activations=False)
    for k in g1:
        np.testing.assert_allclose(g1[k], g2[k], rtol=1e-13, atol=1e-13)


STACK = workloads.StackShape(seed_base=94000, layer=TINY_LLAMA.with_(B=1, T=10), L=2, V=11)


def _stack_case(st, keep=None):
    ls = st.layer
    t = workloads.stack_tensors(st)
    layers = [big_weights(ls, st.seed_base + 100 * (l + 1)) for l in range(st.L)]
    E = t["E"].astype(np.float64) * 20
    w_lm = t["w_lm"].astype(np.float64) * 20
    keep = t["keep"] if keep is None else keep
    return t, layers, E, w_lm, keep


def test_stack_matches_autograd_of_surrogate():
    st = STACK
    ls = st.layer
    t, layers, E, w_lm, keep = _stack_case(st)
    z, saved = ost.stack_forward(t["ids"], E, layers, t["normf_w"], w_lm, ls, round_saved=False)
    g = ost.stack_backward(z, t["targets"], t["ids"], saved, layers, t["normf_w"], w_lm, ls, st.V, keep)
    tl = [_t(w) for w in layers]
    tE = torch.tensor(E, requires_grad=True)
    tnf = torch.tensor(t["normf_w"].astype(np.float64), requires_grad=True)
    tlm = torch.tensor(w_lm.astype(np.float64), requires_grad=True)
    loss = sg.stack_loss(torch.tensor(t["ids"]).long(), torch.tensor(t["targets"]).long(), tE, tl, tnf, tlm,
                         ls, keep=torch.tensor(keep != 0))
    loss.backward()
    assert _rel(g["dw_lm"], tlm.grad.numpy()) < 1e-11
    assert _rel(g["dnormf_w"], tnf.grad.numpy()) < 1e-11
    assert _rel(g["dE"], tE.grad.numpy()) < 1e-11
    for l in range(st.L):
        for name, tt in tl[l].items():
            assert _rel(g["blocks"][l]["d" + name], tt.grad.numpy()) < 1e-10, (l, name)


def test_stack_invariants():
    st = STACK
    ls = st.layer
    t, layers, E, w_lm, keep = _stack_case(st)
    z, saved = ost.stack_forward(t["ids"], E, layers, t["normf_w"], w_lm, ls, round_saved=True)
    g = ost.stack_backward(z, t["targets"], t["ids"], saved, layers, t["normf_w"], w_lm, ls, st.V, keep)
    km = keep.reshape(-1) != 0
    assert np.all(g["dx0"][~km] == 0)
    for gb in g["blocks"]:
        assert np.all(gb["dx"][~km] == 0)
    # dE rows only at kept tokens' ids
    assert set(np.flatnonzero(np.abs(g["dE"]).sum(1))) <= set(t["ids"][km].tolist())
    g0 = ost.stack_backward(z, t["targets"], t["ids"], saved, layers, t["normf_w"], w_lm, ls, st.V,
                            np.zeros_like(keep))
    assert np.all(g0["dw_lm"] == 0) and np.all(g0["dE"] == 0)


def test_stack_streamed_blocks_and_pool_give_the_same_gradients():
    """The full-size stack comparison hands the oracle its saved sets one block
    at a time, takes each block's gradients through on_block, and spreads the
    attention loop over a spawned pool; none of that changes the result."""
    import multiprocessing as mp
    st = STACK
    ls = st.layer
    t, layers, E, w_lm, keep = _stack_case(st)
    z, saved = ost.stack_forward(t["ids"], E, layers, t["normf_w"], w_lm, ls, round_saved=True)
    g = ost.stack_backward(z, t["targets"], t["ids"], saved, layers, t["normf_w"], w_lm, ls, st.V, keep)
    asked = []

    class Lazy:
        def __getitem__(self, l):
            asked.append(l)
            return saved["blocks"][l]

    got = {}
    with mp.get_context("spawn").Pool(2) as pool:
        g2 = ost.stack_backward(z, t["targets"], t["ids"], dict(saved, blocks=Lazy()), layers, t["normf_w"],
                                w_lm, ls, st.V, keep, pool=pool, on_block=lambda l, gb: got.setdefault(l, gb))
    assert asked == list(reversed(range(st.L)))
    for k in ("dw_lm", "dnormf_w", "dE", "dx0"):
        assert _rel(g[k], g2[k]) < 1e-13, k
    for l in range(st.L):
        for k, v in g["blocks"][l].items():
            assert _rel(v, got[l][k]) < 1e-13, (l, k)
