"""Pins for oracle.compaction: a hand-worked fixture, brute force, edge cases."""
import os

import numpy as np
import pytest

from oracle.compaction import compact
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden", "compact_example.txt")


def _read_fixture(path):
    d = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *vals = line.split()
        d[k] = [int(v) for v in vals]
    return d


def test_hand_worked_fixture():
    d = _read_fixture(GOLD)
    B, T = d["B"][0], d["T"][0]
    mask = np.array(d["mask"], dtype=np.uint8).reshape(B, T)
    idx, cu, n = compact(mask)
    assert idx.tolist() == d["idx"]
    assert cu.tolist() == d["cu_kept"]
    assert n == d["n_kept"][0]


def _brute(mask):
    B, T = mask.shape
    idx, cu = [], [0]
    for b in range(B):
        for t in range(T):
            if mask[b, t]:
                idx.append(b * T + t)
        cu.append(len(idx))
    return idx, cu


@pytest.mark.parametrize("B,T,f,kind", [(1, 128, 0.4, "gumbel"), (3, 37, 0.2, "gumbel"),
                                        (4, 64, 0.6, "span"), (2, 1, 0.0, "gumbel")])
def test_brute_force(B, T, f, kind):
    mask = workloads.keep_mask(B, T, f, kind, seed=7)
    idx, cu, n = compact(mask)
    bi, bc = _brute(mask)
    assert idx.tolist() == bi and cu.tolist() == bc and n == len(bi)
    assert idx.dtype == np.int32 and cu.dtype == np.int32


def test_edges():
    idx, cu, n = compact(np.zeros((2, 5), np.uint8))
    assert n == 0 and idx.size == 0 and cu.tolist() == [0, 0, 0]
    idx, cu, n = compact(np.ones((2, 5), np.uint8))
    assert idx.tolist() == list(range(10)) and cu.tolist() == [0, 5, 10]
    # any nonzero byte means kept
    idx, _, _ = compact(np.array([[0, 7, 255, 0]], np.uint8))
    assert idx.tolist() == [1, 2]


def test_mask_generators_filter_exact_count():
    for kind in ("gumbel", "span"):
        for f in (0.0, 0.2, 0.4, 0.6):
            m = workloads.keep_mask(3, 200, f, kind, seed=11)
            nf = workloads.n_filtered(200, f)
            assert (m.sum(axis=1) == 200 - nf).all()
    # floor, not round: 40% of 128 -> 51 filtered, 77 kept
    assert workloads.n_filtered(128, 0.4) == 51
