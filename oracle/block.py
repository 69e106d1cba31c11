"""Decoder block: dense forward (producing the saved set) and Collider's
filtered backward, float64 (test infrastructure only).

Collider (abstract; TL;DR: activation filtering in the backward of every layer)
keeps the forward dense and, in backward, drops the activations and output
gradients of filtered tokens in every layer.  Here that is done full-size:
every saved row and every incoming-gradient row of a filtered token is
replaced by 0 (np.where), the ordinary dense backward is run, and attention
uses the filtered probabilities of :mod:`oracle.attention`.

Shapes (M = B*T tokens): x [M, D]; weights stored [in, out].  ``w`` holds
norm1_w (and norm1_b for LayerNorm), w_qkv [D, (H+2Hkv)dh] with columns
[q heads | k heads | v heads], optional b_qkv, w_o [H*dh, D], optional b_o,
norm2_w (llama), w_up [D, 2F] = [gate | up] (SwiGLU) or [D, F] (fc1, GELU),
optional b_up, w_down [F, D], optional b_down.

Saved set (what the backward reads), rounded to its storage type when it is
produced (bf16; fp32 for lse, mean, rstd) if ``round_saved``:
  llama: x, a = norm1(x), rstd1, qkv (q and k after RoPE), o, lse [B,H,T],
         h = x + attn, b = norm2(h), rstd2, gu = [g | u], s = silu(g)*u
  phi:   x, a = LN(x), mean1, rstd1, qkv (rotated), o, lse, f1 (fc1 pre-GELU)
"""
from __future__ import annotations

import numpy as np

from . import ops
from .attention import attention_forward, filtered_attention_backward


def _split_qkv(qkv, s):
    M = qkv.shape[0]
    nq, nk = s.H * s.dh, s.Hkv * s.dh
    q = qkv[:, :nq].reshape(M, s.H, s.dh)
    k = qkv[:, nq:nq + nk].reshape(M, s.Hkv, s.dh)
    v = qkv[:, nq + nk:].reshape(M, s.Hkv, s.dh)
    return q, k, v


def positions(s):
    """Original position of each token inside its sequence."""
    return np.tile(np.arange(s.T), s.B)


def block_forward(x, w, s, round_saved=True):
    """Dense forward of one block.  Returns (out, saved)."""
    R = ops.to_bf16 if round_saved else (lambda t: np.asarray(t, dtype=np.float64))
    R32 = ops.to_f32 if round_saved else (lambda t: np.asarray(t, dtype=np.float64))
    f64 = lambda t: np.asarray(t, dtype=np.float64)
    x = f64(x)
    pos = positions(s)
    scale = 1.0 / np.sqrt(s.dh)
    sv = dict(x=x)
    if s.norm == "rms":
        rstd1 = R32(1.0 / np.sqrt(np.mean(x * x, axis=-1) + s.eps))
        a = R(x * rstd1[:, None] * f64(w["norm1_w"])[None, :])
        sv.update(rstd1=rstd1)
    else:
        mu = np.mean(x, axis=-1)
        rstd1 = R32(1.0 / np.sqrt(np.mean((x - mu[:, None]) ** 2, axis=-1) + s.eps))
        mu = R32(mu)
        a = R((x - mu[:, None]) * rstd1[:, None] * f64(w["norm1_w"])[None, :] + f64(w["norm1_b"])[None, :])
        sv.update(mean1=mu, rstd1=rstd1)
    sv["a"] = a
    qkv = a @ f64(w["w_qkv"])
    if "b_qkv" in w:
        qkv = qkv + f64(w["b_qkv"])[None, :]
    q, k, v = _split_qkv(R(qkv), s)
    q = R(ops.rope_forward(q, pos, s.rotary_dim, s.rope_base))
    k = R(ops.rope_forward(k, pos, s.rotary_dim, s.rope_base))
    M = x.shape[0]
    sv["qkv"] = np.concatenate([q.reshape(M, -1), k.reshape(M, -1), v.reshape(M, -1)], axis=1)
    o, lse = attention_forward(q, k, v, s.B, s.T, scale)
    o = R(o.reshape(M, -1))
    sv.update(o=o, lse=R32(lse))
    attn = o @ f64(w["w_o"])
    if "b_o" in w:
        attn = attn + f64(w["b_o"])[None, :]
    if s.arch == "llama":
        h = R(x + attn)
        rstd2 = R32(1.0 / np.sqrt(np.mean(h * h, axis=-1) + s.eps))
        b = R(h * rstd2[:, None] * f64(w["norm2_w"])[None, :])
        gu = R(b @ f64(w["w_up"]))
        F = s.F
        sact = R(ops.swiglu_forward(gu[:, :F], gu[:, F:]))
        out = R(h + sact @ f64(w["w_down"]))
        sv.update(h=h, b=b, rstd2=rstd2, gu=gu, s=sact)
    else:
        f1 = a @ f64(w["w_up"])
        if "b_up" in w:
            f1 = f1 + f64(w["b_up"])[None, :]
        f1 = R(f1)
        f2 = R(ops.gelu_tanh_forward(f1))
        mlp = f2 @ f64(w["w_down"])
        if "b_down" in w:
            mlp = mlp + f64(w["b_down"])[None, :]
        out = R(x + attn + mlp)
        sv.update(f1=f1)
    return out, sv


def block_backward(dout, saved, w, s, keep, filter_activations=True, pool=None):
    """Collider filtered backward of one block, full-size and masked.

    keep: [B, T] keep-mask.  Returns a dict of gradients: dx [M, D] (filtered
    rows exactly 0) and fp64 weight gradients named d<weight>.

    filter_activations=False is the prior art Collider improves on (Fig. 2b,
    Fig. 3): only the loss of filtered tokens is dropped, the saved
    activations and the softmax stay dense, so gradients reach filtered rows.
    pool: optional process pool for the attention's (sequence, head) loop.
    """
    keep = np.asarray(keep) != 0
    km = keep.reshape(-1)
    Z = (lambda t: ops.rows_where(km, t)) if filter_activations else \
        (lambda t: np.asarray(t, dtype=np.float64))
    f64 = lambda t: np.asarray(t, dtype=np.float64)
    pos = positions(s)
    scale = 1.0 / np.sqrt(s.dh)
    M = km.size
    g = {}
    dout = Z(dout)
    x = Z(saved["x"])
    a = Z(saved["a"])
    rstd1 = Z(saved["rstd1"])
    qkv = Z(saved["qkv"])
    o = Z(saved["o"])
    lse = f64(saved["lse"])

    if s.arch == "llama":
        h, b, gu, sact = Z(saved["h"]), Z(saved["b"]), Z(saved["gu"]), Z(saved["s"])
        rstd2 = Z(saved["rstd2"])
        F = s.F
        # MLP down: dW_down = s^T dout, ds = dout W_down^T
        g["dw_down"] = sact.T @ dout
        ds = dout @ f64(w["w_down"]).T
        dgate, dup = ops.swiglu_backward(ds, gu[:, :F], gu[:, F:])
        dgu = np.concatenate([dgate, dup], axis=1)
        g["dw_up"] = b.T @ dgu
        db_ = dgu @ f64(w["w_up"]).T
        dhn, g["dnorm2_w"] = ops.rmsnorm_backward(db_, h, rstd2, f64(w["norm2_w"]))
        dh = dout + dhn
        dattn = dh
    else:
        f1 = Z(saved["f1"])
        f2 = ops.gelu_tanh_forward(f1)
        g["dw_down"] = f2.T @ dout
        if "b_down" in w:
            g["db_down"] = dout.sum(axis=0)
        df2 = dout @ f64(w["w_down"]).T
        df1 = ops.gelu_tanh_backward(df2, f1)
        g["dw_up"] = a.T @ df1
        if "b_up" in w:
            g["db_up"] = df1.sum(axis=0)
        da_mlp = df1 @ f64(w["w_up"]).T
        dattn = dout

    # attention output projection
    g["dw_o"] = o.T @ dattn
    if "b_o" in w:
        g["db_o"] = dattn.sum(axis=0)
    do = (dattn @ f64(w["w_o"]).T).reshape(M, s.H, s.dh)
    q, k, v = _split_qkv(qkv, s)
    if filter_activations:
        dq, dk, dv = filtered_attention_backward(q, k, v, do, lse, keep, scale, pool=pool)
    else:
        dq, dk, dv = filtered_attention_backward(q, k, v, do, lse, np.ones_like(keep), scale, pool=pool)
    dq = ops.rope_backward(dq, pos, s.rotary_dim, s.rope_base)
    dk = ops.rope_backward(dk, pos, s.rotary_dim, s.rope_base)
    dqkv = np.concatenate([dq.reshape(M, -1), dk.reshape(M, -1), dv.reshape(M, -1)], axis=1)
    g["dw_qkv"] = a.T @ dqkv
    if "b_qkv" in w:
        g["db_qkv"] = dqkv.sum(axis=0)
    da = dqkv @ f64(w["w_qkv"]).T

    if s.arch == "llama":
        dxn, g["dnorm1_w"] = ops.rmsnorm_backward(da, x, rstd1, f64(w["norm1_w"]))
        g["dx"] = dh + dxn
    else:
        da = da + da_mlp
        mean1 = Z(saved["mean1"])
        dxn, g["dnorm1_w"], g["dnorm1_b"] = ops.layernorm_backward(da, x, mean1, rstd1, f64(w["norm1_w"]))
        g["dx"] = dout + dxn
    if filter_activations:
        g["dx"] = Z(g["dx"])
    return g
