"""Token-wise pieces of the oracle, float64 (test infrastructure only).

Every backward here is the textbook derivative of the forward written beside
it; the Collider-specific part is only the masking of filtered rows, which
the callers apply (abstract: activations of filtered tokens are filtered in
every layer).  Pinned by finite differences in tests/test_oracle_ops.py.
"""
from __future__ import annotations

import math

import numpy as np


# --------------------------------------------------------------------------
# storage rounding used when the oracle's forward writes its saved tensors
# --------------------------------------------------------------------------
def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits, ties
    to even), returned as float64.  Direct from float64, no double rounding."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2**e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0) / 256.0     # 8 significant bits, rint = ties-to-even
    return np.ldexp(r, e)


def to_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def rows_where(keep_rows: np.ndarray, t: np.ndarray) -> np.ndarray:
    """Zero the rows of filtered tokens (keep_rows: [M] bool), NaN-proof."""
    t = np.asarray(t, dtype=np.float64)
    k = keep_rows.reshape((-1,) + (1,) * (t.ndim - 1))
    return np.where(k, t, 0.0)


# --------------------------------------------------------------------------
# linear layer, Y = X W (+ b), W stored [in, out]
# --------------------------------------------------------------------------
def linear_backward(X, W, dY, keep_rows, want_bias=False):
    """Filtered linear backward (abstract: dimension-reduced GEMM reaches the
    sparse result).  Full-size and masked:
        dX = (m*dY) W^T          (filtered rows exactly 0)
        dW = (m*X)^T (m*dY)
        db = sum_rows (m*dY)
    """
    Xm = rows_where(keep_rows, X)
    dYm = rows_where(keep_rows, dY)
    W = np.asarray(W, dtype=np.float64)
    dX = dYm @ W.T
    dW = Xm.T @ dYm
    db = dYm.sum(axis=0) if want_bias else None
    return dX, dW, db


# --------------------------------------------------------------------------
# norms
# --------------------------------------------------------------------------
def rmsnorm_forward(x, gamma, eps):
    x = np.asarray(x, dtype=np.float64)
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)
    return x * rstd[:, None] * gamma[None, :], rstd


def rmsnorm_backward(dy, x, rstd, gamma):
    """y = x*r*gamma, r = (mean(x^2)+eps)^-1/2 with r taken from the forward.
    dx = r*(dy*gamma - xh*mean(dy*gamma*xh)), xh = x*r;  dgamma = sum dy*xh."""
    dy = np.asarray(dy, dtype=np.float64)
    xh = np.asarray(x, dtype=np.float64) * np.asarray(rstd, dtype=np.float64)[:, None]
    g = dy * gamma[None, :]
    c = np.mean(g * xh, axis=-1)
    dx = np.asarray(rstd)[:, None] * (g - xh * c[:, None])
    dgamma = np.sum(dy * xh, axis=0)
    return dx, dgamma


def layernorm_forward(x, gamma, beta, eps):
    x = np.asarray(x, dtype=np.float64)
    mu = np.mean(x, axis=-1)
    var = np.mean((x - mu[:, None]) ** 2, axis=-1)
    rstd = 1.0 / np.sqrt(var + eps)
    return (x - mu[:, None]) * rstd[:, None] * gamma[None, :] + beta[None, :], mu, rstd


def layernorm_backward(dy, x, mean, rstd, gamma):
    """y = xh*gamma + beta, xh = (x-mu)*r.
    dx = r*(g - mean(g) - xh*mean(g*xh)), g = dy*gamma;
    dgamma = sum dy*xh;  dbeta = sum dy."""
    dy = np.asarray(dy, dtype=np.float64)
    xh = (np.asarray(x, dtype=np.float64) - np.asarray(mean)[:, None]) * np.asarray(rstd)[:, None]
    g = dy * gamma[None, :]
    dx = np.asarray(rstd)[:, None] * (g - g.mean(axis=-1, keepdims=True)
                                      - xh * np.mean(g * xh, axis=-1, keepdims=True))
    return dx, np.sum(dy * xh, axis=0), np.sum(dy, axis=0)


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------
def sigmoid(x):
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def swiglu_forward(g, u):
    """s = silu(g) * u, silu(g) = g*sigmoid(g)."""
    return g * sigmoid(g) * u


def swiglu_backward(ds, g, u):
    """dg = ds*u*sig(g)*(1 + g*(1-sig(g))),  du = ds*silu(g)."""
    sg = sigmoid(g)
    return ds * u * sg * (1.0 + g * (1.0 - sg)), ds * g * sg


_GELU_C = math.sqrt(2.0 / math.pi)
_GELU_A = 0.044715


def gelu_tanh_forward(x):
    return 0.5 * x * (1.0 + np.tanh(_GELU_C * (x + _GELU_A * x ** 3)))


def gelu_tanh_backward(dy, x):
    """d/dx of 0.5 x (1 + tanh(c(x + a x^3)))."""
    t = np.tanh(_GELU_C * (x + _GELU_A * x ** 3))
    return dy * (0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * _GELU_C * (1.0 + 3.0 * _GELU_A * x * x))


# --------------------------------------------------------------------------
# rotary position embedding, rotate-half pairing (i, i + r/2) on the first r dims
# --------------------------------------------------------------------------
def rope_angles(pos, rotary_dim, base):
    """theta_i = base^(-2i/r), angle[p, i] = p*theta_i, i < r/2."""
    half = rotary_dim // 2
    inv = base ** (-(2.0 * np.arange(half, dtype=np.float64)) / rotary_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]


def rope_forward(x, pos, rotary_dim, base):
    """x: [M, nheads, dh].  First half / second half of the rotary dims rotate
    as a pair; dims >= rotary_dim pass through."""
    x = np.asarray(x, dtype=np.float64)
    ang = rope_angles(pos, rotary_dim, base)[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    h = rotary_dim // 2
    y = x.copy()
    x1, x2 = x[..., :h], x[..., h:rotary_dim]
    y[..., :h] = x1 * c - x2 * s
    y[..., h:rotary_dim] = x2 * c + x1 * s
    return y


def rope_backward(dy, pos, rotary_dim, base):
    """Transpose of the rotation: rotate the gradient by -angle."""
    dy = np.asarray(dy, dtype=np.float64)
    ang = rope_angles(pos, rotary_dim, base)[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    h = rotary_dim // 2
    dx = dy.copy()
    d1, d2 = dy[..., :h], dy[..., h:rotary_dim]
    dx[..., :h] = d1 * c + d2 * s
    dx[..., h:rotary_dim] = d2 * c - d1 * s
    return dx


# --------------------------------------------------------------------------
# cross-entropy over kept tokens, mean over the kept count
# --------------------------------------------------------------------------
def ce_loss(z, targets, keep_rows):
    z = np.asarray(z, dtype=np.float64)
    mx = z.max(axis=1, keepdims=True)
    lse = (mx[:, 0] + np.log(np.exp(z - mx).sum(axis=1)))
    nll = lse - z[np.arange(z.shape[0]), targets]
    nk = int(np.count_nonzero(keep_rows))
    return float(np.where(keep_rows, nll, 0.0).sum() / max(nk, 1))


def ce_backward(z, targets, keep_rows):
    """dz_i = m_i * (softmax(z_i) - onehot(t_i)) / n_kept (backward token
    filtering of the loss, Fig. 2b).  Filtered rows exactly 0."""
    z = rows_where(keep_rows, z)
    mx = z.max(axis=1, keepdims=True)
    p = np.exp(z - mx)
    p /= p.sum(axis=1, keepdims=True)
    p[np.arange(z.shape[0]), targets] -= 1.0
    nk = int(np.count_nonzero(keep_rows))
    return rows_where(keep_rows, p / max(nk, 1))
