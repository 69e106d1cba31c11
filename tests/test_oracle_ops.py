"""Pins for oracle.ops: central finite differences of the masked loss
L = sum_i m_i <dY_i, Y_i> (token-wise ops: exact), closed forms, rounding."""
import math

import numpy as np
import pytest

from oracle import ops

H = 1e-6


def _fd(fun, x, coords, h=H):
    out = []
    for c in coords:
        xp = x.copy(); xp[c] += h
        xm = x.copy(); xm[c] -= h
        out.append((fun(xp) - fun(xm)) / (2 * h))
    return np.array(out)


def _coords(shape, n, rng):
    return [tuple(int(rng.integers(0, s)) for s in shape) for _ in range(n)]


def _close(a, b, tol=1e-6):
    a, b = np.asarray(a), np.asarray(b)
    assert np.max(np.abs(a - b)) <= tol * max(1.0, np.max(np.abs(b))), (a, b)


def test_linear_backward_fd():
    rng = np.random.default_rng(0)
    M, K, N = 9, 5, 7
    X, W, dY = rng.normal(size=(M, K)), rng.normal(size=(K, N)), rng.normal(size=(M, N))
    b = rng.normal(size=N)
    m = rng.random(M) < 0.6
    loss = lambda X_, W_, b_: float(np.sum(np.where(m[:, None], dY * (X_ @ W_ + b_), 0.0)))
    dX, dW, db = ops.linear_backward(X, W, dY, m, want_bias=True)
    cs = _coords(X.shape, 12, rng)
    _close([dX[c] for c in cs], _fd(lambda t: loss(t, W, b), X, cs))
    cs = _coords(W.shape, 12, rng)
    _close([dW[c] for c in cs], _fd(lambda t: loss(X, t, b), W, cs))
    _close(db, _fd(lambda t: loss(X, W, t), b, [(i,) for i in range(N)]))
    assert np.all(dX[~m] == 0)


def test_linear_backward_poison_invariance():
    rng = np.random.default_rng(1)
    M, K, N = 6, 4, 3
    X, W, dY = rng.normal(size=(M, K)), rng.normal(size=(K, N)), rng.normal(size=(M, N))
    m = np.array([1, 0, 1, 1, 0, 1], bool)
    a = ops.linear_backward(X, W, dY, m)
    X2, dY2 = X.copy(), dY.copy()
    X2[~m] = np.nan; dY2[~m] = np.inf
    b = ops.linear_backward(X2, W, dY2, m)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("norm", ["rms", "ln"])
def test_norm_backward_fd(norm):
    rng = np.random.default_rng(2)
    M, D, eps = 5, 8, 1e-5
    x, dy = rng.normal(size=(M, D)), rng.normal(size=(M, D))
    gamma, beta = 1 + 0.3 * rng.normal(size=D), 0.3 * rng.normal(size=D)
    if norm == "rms":
        fwd = lambda x_, g_: ops.rmsnorm_forward(x_, g_, eps)[0]
        _, r = ops.rmsnorm_forward(x, gamma, eps)
        dx, dg = ops.rmsnorm_backward(dy, x, r, gamma)
    else:
        fwd = lambda x_, g_: ops.layernorm_forward(x_, g_, beta, eps)[0]
        _, mu, r = ops.layernorm_forward(x, gamma, beta, eps)
        dx, dg, dbeta = ops.layernorm_backward(dy, x, mu, r, gamma)
        _close(dbeta, dy.sum(0))
    loss = lambda x_, g_: float(np.sum(dy * fwd(x_, g_)))
    cs = _coords(x.shape, 15, rng)
    _close([dx[c] for c in cs], _fd(lambda t: loss(t, gamma), x, cs))
    _close(dg, _fd(lambda t: loss(x, t), gamma, [(i,) for i in range(D)]))


def test_activation_backward_fd():
    rng = np.random.default_rng(3)
    g, u, ds = rng.normal(size=20) * 3, rng.normal(size=20), rng.normal(size=20)
    dg, du = ops.swiglu_backward(ds, g, u)
    e = np.eye(20)
    fd_g = [(np.sum(ds * ops.swiglu_forward(g + H * e[i], u)) - np.sum(ds * ops.swiglu_forward(g - H * e[i], u))) / (2 * H) for i in range(20)]
    fd_u = [(np.sum(ds * ops.swiglu_forward(g, u + H * e[i])) - np.sum(ds * ops.swiglu_forward(g, u - H * e[i]))) / (2 * H) for i in range(20)]
    _close(dg, fd_g); _close(du, fd_u)
    x = rng.normal(size=20) * 3
    dx = ops.gelu_tanh_backward(ds, x)
    fd = [(np.sum(ds * ops.gelu_tanh_forward(x + H * e[i])) - np.sum(ds * ops.gelu_tanh_forward(x - H * e[i]))) / (2 * H) for i in range(20)]
    _close(dx, fd)
    # closed forms: silu(0) = 0, d silu(0) = 1/2; gelu(0)' = 1/2
    assert ops.swiglu_backward(np.array([1.0]), np.array([0.0]), np.array([1.0]))[0][0] == 0.5
    assert ops.gelu_tanh_backward(np.array([1.0]), np.array([0.0]))[0] == 0.5


@pytest.mark.parametrize("r,dh", [(8, 8), (4, 8)])
def test_rope_backward_fd_and_orthogonality(r, dh):
    rng = np.random.default_rng(4)
    M, nh = 6, 3
    pos = rng.integers(0, 5000, size=M)
    x, dy = rng.normal(size=(M, nh, dh)), rng.normal(size=(M, nh, dh))
    dx = ops.rope_backward(dy, pos, r, 10000.0)
    loss = lambda t: float(np.sum(dy * ops.rope_forward(t, pos, r, 10000.0)))
    cs = _coords(x.shape, 20, rng)
    _close([dx[c] for c in cs], _fd(loss, x, cs))
    # rotation is orthogonal: backward inverts forward; norm preserved
    _close(ops.rope_backward(ops.rope_forward(x, pos, r, 10000.0), pos, r, 10000.0), x, 1e-12)
    # position 0 is the identity; dims >= r pass through
    _close(ops.rope_forward(x, np.zeros(M, int), r, 10000.0), x, 0)
    assert np.array_equal(ops.rope_forward(x, pos, r, 10000.0)[..., r:], x[..., r:])
    # closed form, r=2 pair: angle = pos * base^0 = pos
    y = ops.rope_forward(np.array([[[1.0, 0.0]]]), np.array([1]), 2, 10000.0)
    _close(y[0, 0], [math.cos(1.0), math.sin(1.0)], 1e-15)


def test_ce_backward_fd():
    rng = np.random.default_rng(5)
    M, V = 7, 11
    z, t = rng.normal(size=(M, V)) * 2, rng.integers(0, V, size=M)
    m = np.array([1, 1, 0, 1, 0, 1, 1], bool)
    dz = ops.ce_backward(z, t, m)
    cs = _coords(z.shape, 25, rng)
    _close([dz[c] for c in cs], _fd(lambda q: ops.ce_loss(q, t, m), z, cs))
    assert np.all(dz[~m] == 0)
    # rows of softmax - onehot sum to 0
    _close(dz.sum(axis=1), np.zeros(M), 1e-15)
    # closed form: uniform logits, one kept token -> (1/V - onehot)
    dz1 = ops.ce_backward(np.zeros((2, 4)), np.array([2, 0]), np.array([True, False]))
    _close(dz1[0], [0.25, 0.25, -0.75, 0.25], 1e-15)


def test_bf16_rounding_closed_forms():
    v = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -7, -(1 + 2 ** -8), 3.0, 0.0,
                  1 + 2 ** -8 + 2 ** -20])
    want = np.array([1.0, 1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0, 3.0, 0.0, 1 + 2 ** -7])
    assert np.array_equal(ops.to_bf16(v), want)
    # agrees with torch's own fp32 -> bf16 conversion on ordinary values
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(6).normal(size=1000).astype(np.float32)
    tb = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ops.to_bf16(x.astype(np.float64)), tb)
