"""Causal GQA attention: dense forward and Collider's filtered backward.
Float64, one (sequence, head) at a time (test infrastructure only).

Layouts: q [M, H, dh], k and v [M, Hkv, dh], M = B*T tokens in sequence
order; query head h reads kv head floor(h*Hkv/H); lse [B, H, T] natural log.

Filtered backward (Collider, Fig. 3 and Fig. 5 captions): leaving the softmax
of filtered tokens unchanged makes G_V dense and spreads density to every
earlier layer, so the probabilities are filtered too, and the same filtered
probabilities serve the Q and K gradients.  Readings taken here where the
pages are silent:
  * P is recomputed from the dense forward's logsumexp, P_ij = exp(S_ij -
    lse_i) on causal pairs (original positions), with no renormalisation over
    the kept keys.
  * P'_ij = m_i m_j P_ij (filtered query rows and key columns zeroed).
  * the softmax-backward correction term is taken over P':
    D_i = sum_j P'_ij dP_ij.
  * dS = P' * (dP - D);  dQ = dS K s;  dK = dS^T Q s;  G_V = P'^T dO;
    s = the logit scale.  GQA sums dK and dV over each group of query heads.
"""
from __future__ import annotations

import numpy as np


def _kv_head(h, H, Hkv):
    return (h * Hkv) // H


def attention_forward(q, k, v, B, T, scale, causal=True):
    """Dense forward.  Returns o [M, H, dh] and lse [B, H, T]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    M, H, dh = q.shape
    Hkv = k.shape[1]
    o = np.zeros_like(q)
    lse = np.zeros((B, H, T))
    allowed = np.tril(np.ones((T, T), dtype=bool)) if causal else np.ones((T, T), dtype=bool)
    for b in range(B):
        rows = slice(b * T, (b + 1) * T)
        for h in range(H):
            hk = _kv_head(h, H, Hkv)
            S = (q[rows, h, :] @ k[rows, hk, :].T) * scale
            S = np.where(allowed, S, -np.inf)
            mx = S.max(axis=1, keepdims=True)
            l = mx[:, 0] + np.log(np.exp(S - mx).sum(axis=1))
            P = np.exp(S - l[:, None])
            o[rows, h, :] = P @ v[rows, hk, :]
            lse[b, h, :] = l
    return o, lse


def _head_backward(task):
    """One (sequence, query head): the filtered backward of that head alone.
    Returns its dQ rows and its contributions to dK, dV of the head's kv head."""
    Q, K, V, G, lse_row, mi, causal, zero_p, scale = task
    T = mi.size
    pos = np.arange(T)
    allowed = (pos[None, :] <= pos[:, None]) if causal else np.ones((T, T), dtype=bool)
    pair = np.outer(mi, mi) if zero_p else np.ones((T, T), dtype=bool)
    S = (Q @ K.T) * scale
    P = np.where(allowed, np.exp(np.where(allowed, S, 0.0) - lse_row[:, None]), 0.0)
    Pf = np.where(pair, P, 0.0)                 # P'
    dv = Pf.T @ G                               # G_V
    dP = G @ V.T
    D = np.sum(Pf * dP, axis=1)                 # over the filtered P'
    dS = Pf * (dP - D[:, None])
    return (dS @ K) * scale, (dS.T @ Q) * scale, dv


def filtered_attention_backward(q, k, v, dO, lse, keep, scale, causal=True, zero_p=True, pool=None):
    """Collider attention backward, full-size and masked.

    keep: [B, T] keep-mask.  Rows of q, k, v, dO of filtered tokens are
    replaced by 0 first (np.where: arbitrary values cannot leak), and so is
    lse at filtered query positions.  zero_p=False is the ablation of Fig. 3:
    the softmax of filtered tokens is left as the dense forward made it (K, V
    of filtered tokens kept, P not zeroed), only the upstream gradient rows
    are filtered, and G_V picks up rows at filtered tokens.
    pool: an optional process pool (anything with ``map``) over which the
    independent (sequence, head) computations are spread; the results are
    summed in the same order either way.
    Returns dq [M, H, dh], dk and dv [M, Hkv, dh].
    """
    keep = np.asarray(keep) != 0
    B, T = keep.shape
    km = keep.reshape(-1)
    act = km if zero_p else np.ones_like(km)      # the ablation keeps K, V of filtered tokens
    q = np.where(km[:, None, None], np.asarray(q, dtype=np.float64), 0.0)
    k = np.where(act[:, None, None], np.asarray(k, dtype=np.float64), 0.0)
    v = np.where(act[:, None, None], np.asarray(v, dtype=np.float64), 0.0)
    dO = np.where(km[:, None, None], np.asarray(dO, dtype=np.float64), 0.0)
    lse = np.where(keep[:, None, :], np.asarray(lse, dtype=np.float64), 0.0)
    M, H, dh = q.shape
    Hkv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        rows = slice(b * T, (b + 1) * T)
        tasks = [(q[rows, h, :], k[rows, _kv_head(h, H, Hkv), :], v[rows, _kv_head(h, H, Hkv), :],
                  dO[rows, h, :], lse[b, h, :], keep[b], causal, zero_p, scale) for h in range(H)]
        outs = (pool.map if pool is not None else map)(_head_backward, tasks)
        for h, (dq_h, dk_h, dv_h) in enumerate(outs):
            hk = _kv_head(h, H, Hkv)
            dq[rows, h, :] = dq_h
            dk[rows, hk, :] += dk_h
            dv[rows, hk, :] += dv_h
    return dq, dk, dv
