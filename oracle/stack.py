"""Decoder stack: token embedding -> L blocks -> final RMSNorm -> untied LM
head -> cross-entropy over kept tokens.  Float64 (test infrastructure only).

Backward token filtering (Collider, Fig. 2b) drops the loss terms of
filtered tokens; Collider then drops their activations in every layer
(abstract), so the same keep-mask applies to the loss and to every block.
The loss is the mean over kept tokens (reading: "cross-entropy over kept
tokens only" averaged by the kept count).
"""
from __future__ import annotations

import numpy as np

from . import ops
from .block import block_forward, block_backward


def stack_forward(ids, E, layers, normf_w, w_lm, ls, round_saved=True):
    """ids [M] int.  Returns (logits z [M, V], saved) where saved holds each
    block's saved set, the final-norm input xL and its rstd, y = norm(xL)."""
    R = ops.to_bf16 if round_saved else (lambda t: np.asarray(t, dtype=np.float64))
    R32 = ops.to_f32 if round_saved else (lambda t: np.asarray(t, dtype=np.float64))
    x = np.asarray(E, dtype=np.float64)[np.asarray(ids)]
    blocks = []
    for w in layers:
        x, sv = block_forward(x, w, ls, round_saved=round_saved)
        blocks.append(sv)
    rstd = R32(1.0 / np.sqrt(np.mean(x * x, axis=-1) + ls.eps))
    y = R(x * rstd[:, None] * np.asarray(normf_w, dtype=np.float64)[None, :])
    z = R(y @ np.asarray(w_lm, dtype=np.float64))
    return z, dict(blocks=blocks, xL=x, rstdf=rstd, y=y)


def stack_backward(z, targets, ids, saved, layers, normf_w, w_lm, ls, V, keep, filter_activations=True,
                   pool=None, on_block=None):
    """Filtered backward of the whole stack.  Returns dict with dz-derived
    dw_lm [D, V], dnormf_w [D], dE [V, D] and per-block gradient dicts
    (``blocks``, input order), plus dx0 (gradient at the embedding output).
    ``saved["blocks"]`` is indexed once per block, top block first, so it may
    produce each block's saved set on demand.  pool: optional process pool
    for the attention loop.  on_block(l, grads), if given, receives each
    block's gradients as soon as they exist, and only dx is kept between
    blocks (the per-block dicts are then not returned)."""
    keep = np.asarray(keep) != 0
    km = keep.reshape(-1)
    Z = (lambda t: ops.rows_where(km, t)) if filter_activations else \
        (lambda t: np.asarray(t, dtype=np.float64))
    out = {}
    dz = ops.ce_backward(z, targets, km)
    y = Z(saved["y"])
    out["dw_lm"] = y.T @ dz
    dy = dz @ np.asarray(w_lm, dtype=np.float64).T
    xL = Z(saved["xL"])
    rstd = Z(saved["rstdf"])
    dx, out["dnormf_w"] = ops.rmsnorm_backward(dy, xL, rstd, np.asarray(normf_w, dtype=np.float64))
    grads = [None] * len(layers)
    for l in reversed(range(len(layers))):
        g = block_backward(dx, saved["blocks"][l], layers[l], ls, keep,
                           filter_activations=filter_activations, pool=pool)
        dx = g["dx"]
        if on_block is not None:
            on_block(l, g)
        else:
            grads[l] = g
    out["blocks"] = grads
    out["dx0"] = dx
    dE = np.zeros((V, dx.shape[1]))
    rows = km if filter_activations else np.ones_like(km)
    np.add.at(dE, np.asarray(ids)[rows], dx[rows])
    out["dE"] = dE
    return out
