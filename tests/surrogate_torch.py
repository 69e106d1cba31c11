"""Float64 torch forward models used to pin the oracle (tests only).

Written independently of ``oracle/``: plain forward definitions whose
autograd gradient the oracle's hand-written backward must reproduce.

The Collider backward is the exact gradient of a *surrogate* forward that
has the same values as the dense forward but lets no gradient reach filtered
tokens through attention:
  * logits of filtered keys are stop-gradient (they still normalise the
    softmax),
  * P @ V splits into (P * m_j) @ V + stopgrad((P * (1 - m_j)) @ V),
  * the loss is masked by m_i.
With ``mask=None`` (or an all-ones mask) this is the plain dense model.
Frozen pieces can be taken from a base evaluation (``frozen``), which makes
finite differences of the surrogate well defined.
"""
from __future__ import annotations

import math

import torch


def rms(x, gamma, eps):
    return x * torch.rsqrt((x * x).mean(-1, keepdim=True) + eps) * gamma


def ln(x, gamma, beta, eps):
    mu = x.mean(-1, keepdim=True)
    var = ((x - mu) ** 2).mean(-1, keepdim=True)
    return (x - mu) / torch.sqrt(var + eps) * gamma + beta


def rope(x, pos, r, base):
    # x [M, nh, dh]; rotate-half pairing on the first r dims
    half = r // 2
    inv = base ** (-(2.0 * torch.arange(half, dtype=torch.float64)) / r)
    ang = pos.to(torch.float64)[:, None] * inv[None, :]
    c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    x1, x2, rest = x[..., :half], x[..., half:r], x[..., r:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s, rest], dim=-1)


def gelu_tanh(x):
    return 0.5 * x * (1 + torch.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))


def attention(q, k, v, B, T, keep, frozen, tag):
    """q [M,H,dh], k/v [M,Hkv,dh]; keep [B,T] bool or None (dense)."""
    M, H, dh = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(dh)
    outs = []
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    for b in range(B):
        rows = slice(b * T, (b + 1) * T)
        heads = []
        for h in range(H):
            hk = (h * Hkv) // H
            S = q[rows, h] @ k[rows, hk].T * scale
            key = (tag, b, h)
            if keep is not None:
                mj = keep[b][None, :]
                Sfz = frozen.setdefault(("S",) + key, S.detach())
                S = torch.where(mj, S, Sfz)
            S = S.masked_fill(~causal, float("-inf"))
            P = torch.softmax(S, dim=-1)
            if keep is not None:
                mjf = keep[b].to(torch.float64)[None, :]
                dead = frozen.setdefault(("PV",) + key, ((P * (1 - mjf)) @ v[rows, hk]).detach())
                o = (P * mjf) @ v[rows, hk] + dead
            else:
                o = P @ v[rows, hk]
            heads.append(o)
        outs.append(torch.stack(heads, dim=1))
    return torch.cat(outs, dim=0)


def block(x, w, s, keep=None, frozen=None, tag=0):
    """One decoder block (llama or phi), float64 torch."""
    frozen = {} if frozen is None else frozen
    M = x.shape[0]
    pos = torch.arange(s.T).repeat(s.B)
    if s.norm == "rms":
        a = rms(x, w["norm1_w"], s.eps)
    else:
        a = ln(x, w["norm1_w"], w["norm1_b"], s.eps)
    qkv = a @ w["w_qkv"]
    if "b_qkv" in w:
        qkv = qkv + w["b_qkv"]
    nq, nk = s.H * s.dh, s.Hkv * s.dh
    q = rope(qkv[:, :nq].reshape(M, s.H, s.dh), pos, s.rotary_dim, s.rope_base)
    k = rope(qkv[:, nq:nq + nk].reshape(M, s.Hkv, s.dh), pos, s.rotary_dim, s.rope_base)
    v = qkv[:, nq + nk:].reshape(M, s.Hkv, s.dh)
    o = attention(q, k, v, s.B, s.T, keep, frozen, tag).reshape(M, -1)
    att = o @ w["w_o"]
    if "b_o" in w:
        att = att + w["b_o"]
    if s.arch == "llama":
        h = x + att
        b = rms(h, w["norm2_w"], s.eps)
        gu = b @ w["w_up"]
        g_, u_ = gu[:, :s.F], gu[:, s.F:]
        return h + (torch.nn.functional.silu(g_) * u_) @ w["w_down"]
    f1 = a @ w["w_up"]
    if "b_up" in w:
        f1 = f1 + w["b_up"]
    mlp = gelu_tanh(f1) @ w["w_down"]
    if "b_down" in w:
        mlp = mlp + w["b_down"]
    return x + att + mlp


def stack_loss(ids, targets, E, layers, normf_w, w_lm, ls, keep=None, frozen=None):
    """Mean cross-entropy over kept tokens of the L-block stack."""
    frozen = {} if frozen is None else frozen
    x = E[ids]
    for l, w in enumerate(layers):
        x = block(x, w, ls, keep=keep, frozen=frozen, tag=l)
    z = rms(x, normf_w, ls.eps) @ w_lm
    nll = torch.nn.functional.cross_entropy(z, targets, reduction="none")
    if keep is None:
        return nll.mean()
    km = keep.reshape(-1)
    return torch.where(km, nll, torch.zeros_like(nll)).sum() / km.sum()
