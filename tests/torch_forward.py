"""A dense block forward written with plain torch ops on the GPU.

Test infrastructure: the full-size stack test needs the saved activations of
22 blocks on the device and also hands them to the fp64 oracle, so they are
produced here, independently of the library under test.
"""
from __future__ import annotations

import math

import torch


def gpu_forward(s, w, x):
    """The saved activations the backward reads, rounded to their storage types.
    Llama-style blocks (RMSNorm, GQA, RoPE, SwiGLU, optional QKV bias) and
    Phi-style parallel blocks (LayerNorm, partial RoPE, GELU-tanh MLP, biases)."""
    dev = x.device
    M = s.M
    f = lambda t: t.float()
    mm = lambda a_, w_: (a_.bfloat16() @ w_.bfloat16()).float()   # bf16 tensor-core matmul
    xf = f(x)
    out = {}
    if s.norm == "ln":
        mean1 = xf.mean(-1)
        rstd1 = torch.rsqrt((xf - mean1[:, None]).pow(2).mean(-1) + s.eps)
        a = ((xf - mean1[:, None]) * rstd1[:, None] * f(w["norm1_w"]) + f(w["norm1_b"])).bfloat16()
        out["mean1"] = mean1
    else:
        rstd1 = torch.rsqrt(xf.pow(2).mean(-1) + s.eps)
        a = (xf * rstd1[:, None] * f(w["norm1_w"])).bfloat16()
    qkv = mm(a, w["w_qkv"])
    if "b_qkv" in w:
        qkv = qkv + f(w["b_qkv"])
    qkv = qkv.bfloat16()
    nq, nk = s.H * s.dh, s.Hkv * s.dh
    pos = torch.arange(s.T, device=dev).repeat(s.B).double()
    half = s.rotary_dim // 2
    inv = s.rope_base ** (-(2.0 * torch.arange(half, device=dev, dtype=torch.float64)) / s.rotary_dim)
    ang = pos[:, None] * inv[None, :]
    cos, sin = torch.cos(ang).float()[:, None, :], torch.sin(ang).float()[:, None, :]

    def rope(t, nh):
        t = f(t).view(M, nh, s.dh)
        x1, x2, rest = t[..., :half], t[..., half:s.rotary_dim], t[..., s.rotary_dim:]
        return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin, rest], -1).bfloat16()

    q = rope(qkv[:, :nq], s.H)
    k = rope(qkv[:, nq:nq + nk], s.Hkv)
    v = qkv[:, nq + nk:].reshape(M, s.Hkv, s.dh)
    qkv_rot = torch.cat([q.reshape(M, -1), k.reshape(M, -1), v.reshape(M, -1)], 1).contiguous()
    o = torch.empty(M, s.H, s.dh, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(s.B, s.H, s.T, dtype=torch.float32, device=dev)
    causal = torch.ones(s.T, s.T, dtype=torch.bool, device=dev).tril()
    G = s.H // s.Hkv
    for b in range(s.B):
        rows = slice(b * s.T, (b + 1) * s.T)
        for h in range(s.H):
            S = f(q[rows, h]) @ f(k[rows, h // G]).T / math.sqrt(s.dh)
            S = S.masked_fill(~causal, float("-inf"))
            l = torch.logsumexp(S, -1)
            o[rows, h] = (torch.exp(S - l[:, None]) @ f(v[rows, h // G])).bfloat16()
            lse[b, h] = l
    o = o.reshape(M, -1)
    if s.arch == "phi":
        f1 = mm(a, w["w_up"])
        if "b_up" in w:
            f1 = f1 + f(w["b_up"])
        out.update(x=x, a=a, rstd1=rstd1, qkv=qkv_rot, o=o, lse=lse, up=f1.bfloat16())
        return out
    h_ = (xf + mm(o, w["w_o"])).bfloat16()
    rstd2 = torch.rsqrt(f(h_).pow(2).mean(-1) + s.eps)
    bn = (f(h_) * rstd2[:, None] * f(w["norm2_w"])).bfloat16()
    gu = mm(bn, w["w_up"]).bfloat16()
    g_, u_ = f(gu[:, :s.F]), f(gu[:, s.F:])
    sact = (g_ * torch.sigmoid(g_) * u_).bfloat16()
    out.update(x=x, a=a, rstd1=rstd1, qkv=qkv_rot, o=o, lse=lse, h=h_, b=bn, rstd2=rstd2, up=gu, s=sact)
    return out
