"""Pins for oracle.attention: a closed-form two-token case, float64 autograd
of the stop-gradient surrogate, finite differences of that surrogate,
0% filtering = plain dense autograd, 100% = zeros, poisoning, the Fig. 3
ablation."""
import math

import numpy as np
import pytest
import torch

from oracle.attention import attention_forward, filtered_attention_backward
import surrogate_torch as sg


def _inputs(B, T, H, Hkv, dh, seed):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(B * T, H, dh))
    k = rng.normal(size=(B * T, Hkv, dh))
    v = rng.normal(size=(B * T, Hkv, dh))
    dO = rng.normal(size=(B * T, H, dh))
    return q, k, v, dO


def _autograd(q, k, v, dO, keep, B, T):
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    kt = None if keep is None else torch.tensor(keep != 0)
    o = sg.attention(tq, tk, tv, B, T, kt, {}, 0)
    m = torch.ones(B * T, dtype=torch.float64) if keep is None else torch.tensor(keep.reshape(-1).astype(np.float64))
    (o * torch.tensor(dO) * m[:, None, None]).sum().backward()
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def test_closed_form_two_tokens():
    # T=2, dh=1, one head; token 0 filtered.  Only the pair (1,1) survives:
    #   lse1 = log(e^{q1 k0} + e^{q1 k1}),  p = e^{q1 k1 - lse1}
    #   dV1 = p dO1,  D1 = p dO1 v1,  dS11 = p (dO1 v1 - D1) = p(1-p) dO1 v1
    #   dq1 = dS11 k1,  dk1 = dS11 q1  (scale 1/sqrt(1) = 1); token 0 all zero
    q = np.array([0.3, 0.8]).reshape(2, 1, 1)
    k = np.array([-0.5, 1.1]).reshape(2, 1, 1)
    v = np.array([2.0, -1.5]).reshape(2, 1, 1)
    dO = np.array([0.7, 1.3]).reshape(2, 1, 1)
    keep = np.array([[0, 1]])
    _, lse = attention_forward(q, k, v, 1, 2, 1.0)
    l1 = math.log(math.exp(0.8 * -0.5) + math.exp(0.8 * 1.1))
    assert abs(lse[0, 0, 1] - l1) < 1e-15 and abs(lse[0, 0, 0] - 0.3 * -0.5) < 1e-15
    dq, dk, dv = filtered_attention_backward(q, k, v, dO, lse, keep, 1.0)
    p = math.exp(0.8 * 1.1 - l1)
    dS = p * (1 - p) * 1.3 * -1.5
    np.testing.assert_allclose(dv.ravel(), [0.0, p * 1.3], rtol=1e-14)
    np.testing.assert_allclose(dq.ravel(), [0.0, dS * 1.1], rtol=1e-14)
    np.testing.assert_allclose(dk.ravel(), [0.0, dS * 0.8], rtol=1e-14)


@pytest.mark.parametrize("B,T,H,Hkv,dh", [(2, 8, 2, 1, 8), (1, 9, 4, 2, 4), (2, 6, 2, 2, 8)])
def test_matches_autograd_of_surrogate(B, T, H, Hkv, dh):
    q, k, v, dO = _inputs(B, T, H, Hkv, dh, seed=B * 100 + T)
    keep = (np.random.default_rng(T).random((B, T)) < 0.6).astype(np.uint8)
    scale = 1 / math.sqrt(dh)
    o, lse = attention_forward(q, k, v, B, T, scale)
    dq, dk, dv = filtered_attention_backward(q, k, v, dO, lse, keep, scale)
    to, tq, tk, tv = _autograd(q, k, v, dO, keep, B, T)
    assert _rel(to, o) < 1e-12          # surrogate forward has the dense values
    assert _rel(dq, tq) < 1e-12 and _rel(dk, tk) < 1e-12 and _rel(dv, tv) < 1e-12


def test_matches_finite_differences_of_surrogate():
    B, T, H, Hkv, dh = 1, 7, 2, 1, 4
    q, k, v, dO = _inputs(B, T, H, Hkv, dh, seed=5)
    keep = np.array([[1, 0, 1, 1, 0, 1, 1]], np.uint8)
    scale = 0.5
    _, lse = attention_forward(q, k, v, B, T, scale)
    dq, dk, dv = filtered_attention_backward(q, k, v, dO, lse, keep, scale)
    kt = torch.tensor(keep != 0)
    m = torch.tensor(keep.reshape(-1).astype(np.float64))[:, None, None]
    frozen = {}
    base = [torch.tensor(a) for a in (q, k, v)]
    sg.attention(*base, B, T, kt, frozen, 0)        # record the frozen pieces

    def L(qq, kk, vv):
        return float((sg.attention(torch.tensor(qq), torch.tensor(kk), torch.tensor(vv), B, T, kt, frozen, 0)
                      * torch.tensor(dO) * m).sum())
    h = 1e-6
    rng = np.random.default_rng(9)
    for which, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(10):
            c = tuple(int(rng.integers(0, s)) for s in arr.shape)

            def shifted(delta):
                args = {"q": q, "k": k, "v": v}
                a2 = arr.copy()
                a2[c] += delta
                args[which] = a2
                return L(args["q"], args["k"], args["v"])
            fd = (shifted(h) - shifted(-h)) / (2 * h)
            assert abs(fd - grad[c]) < 1e-7 * max(1, np.max(np.abs(grad))), (which, c, fd, grad[c])


def test_zero_filtering_is_dense_backward():
    B, T, H, Hkv, dh = 2, 8, 4, 2, 8
    q, k, v, dO = _inputs(B, T, H, Hkv, dh, seed=1)
    scale = 1 / math.sqrt(dh)
    _, lse = attention_forward(q, k, v, B, T, scale)
    dq, dk, dv = filtered_attention_backward(q, k, v, dO, lse, np.ones((B, T)), scale)
    _, tq, tk, tv = _autograd(q, k, v, dO, None, B, T)
    assert _rel(dq, tq) < 1e-12 and _rel(dk, tk) < 1e-12 and _rel(dv, tv) < 1e-12


def test_full_filtering_and_filtered_rows_zero_and_poison():
    B, T, H, Hkv, dh = 2, 8, 2, 1, 8
    q, k, v, dO = _inputs(B, T, H, Hkv, dh, seed=2)
    scale = 1 / math.sqrt(dh)
    _, lse = attention_forward(q, k, v, B, T, scale)
    for r in filtered_attention_backward(q, k, v, dO, lse, np.zeros((B, T)), scale):
        assert np.all(r == 0)
    keep = (np.random.default_rng(3).random((B, T)) < 0.5).astype(np.uint8)
    a = filtered_attention_backward(q, k, v, dO, lse, keep, scale)
    km = keep.reshape(-1) != 0
    for r in a:
        assert np.all(r[~km] == 0)
    q2, k2, v2, d2, l2 = q.copy(), k.copy(), v.copy(), dO.copy(), lse.copy()
    q2[~km] = np.nan; k2[~km] = 1e30; v2[~km] = -np.inf; d2[~km] = np.nan
    l2[np.broadcast_to((keep == 0)[:, None, :], l2.shape)] = np.nan
    b = filtered_attention_backward(q2, k2, v2, d2, l2, keep, scale)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_fig3_ablation_leaves_gv_dense():
    B, T, H, Hkv, dh = 1, 8, 2, 1, 8
    q, k, v, dO = _inputs(B, T, H, Hkv, dh, seed=4)
    scale = 1 / math.sqrt(dh)
    _, lse = attention_forward(q, k, v, B, T, scale)
    keep = np.array([[1, 0, 1, 1, 0, 1, 1, 1]], np.uint8)
    _, _, dv = filtered_attention_backward(q, k, v, dO, lse, keep, scale, zero_p=False)
    _, _, dvf = filtered_attention_backward(q, k, v, dO, lse, keep, scale, zero_p=True)
    filt = keep.reshape(-1) == 0
    assert np.all(np.abs(dv[filt]).max(axis=(1, 2)) > 0)      # G_V no longer sparse
    assert np.all(dvf[filt] == 0)


def test_process_pool_gives_the_sequential_result():
    """Spreading the (sequence, head) loop over a spawned process pool (as the
    full-size stack comparison does) sums the same terms in the same order."""
    import multiprocessing as mp
    rng = np.random.default_rng(3)
    B, T, H, Hkv, dh = 2, 24, 4, 2, 8
    q, k, v, dO = (rng.normal(size=(B * T, n, dh)) for n in (H, Hkv, Hkv, H))
    keep = (rng.random((B, T)) > 0.4).astype(np.uint8)
    _, lse = attention_forward(q, k, v, B, T, 0.35)
    seq = filtered_attention_backward(q, k, v, dO, lse, keep, 0.35)
    with mp.get_context("spawn").Pool(2) as pool:
        par = filtered_attention_backward(q, k, v, dO, lse, keep, 0.35, pool=pool)
    for a, b in zip(seq, par):
        assert np.allclose(a, b, rtol=1e-13, atol=1e-13)
