"""Keep-mask selection and compaction (test infrastructure only).

Collider abstract: the would-be sparse GEMM over all tokens is rewritten as a
dense GEMM whose token dimension is cut down to the kept tokens.  That needs the
list of kept tokens; this is its plain definition: the ascending flat indices
of the nonzero mask entries, the number of kept tokens before each sequence
start, and the total.
"""
from __future__ import annotations

import numpy as np


def compact(keep: np.ndarray):
    """keep: [B, T] (nonzero = kept).  Returns (idx int32 [n_kept], cu_kept
    int32 [B+1], n_kept int).  idx is strictly increasing; cu_kept[b] is the
    number of kept tokens in sequences 0..b-1."""
    keep = np.asarray(keep)
    B, T = keep.shape
    flat = keep.reshape(-1) != 0
    idx = np.flatnonzero(flat).astype(np.int32)
    per_seq = flat.reshape(B, T).sum(axis=1)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(per_seq)
    return idx, cu, int(idx.size)


def select_keep(scores: np.ndarray, n_filter: int) -> np.ndarray:
    """The token filter's decision from per-token scores (Fig. 2b: the loss of
    the filtered tokens is dropped): in every sequence the n_filter lowest
    scores are filtered, equal scores filtered lower position first; NaN
    scores order above every number.  scores [B, T]; returns uint8 [B, T],
    1 = kept."""
    scores = np.asarray(scores, dtype=np.float32)
    B, T = scores.shape
    keep = np.ones((B, T), dtype=np.uint8)
    pos = np.arange(T)
    for b in range(B):
        s = np.where(scores[b] == 0, np.float32(0), scores[b])   # -0.0 ties with +0.0
        order = np.lexsort((pos, s))                            # NaN sorts last
        keep[b, order[:n_filter]] = 0
    return keep
