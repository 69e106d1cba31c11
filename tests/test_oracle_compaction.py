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


def _brute_select(scores, n):
    B, T = scores.shape
    keep = np.ones((B, T), np.uint8)
    for b in range(B):
        def key(p):
            v = float(scores[b, p])
            return (1, 0.0, p) if v != v else (0, v, p)    # NaN after every number
        for p in sorted(range(T), key=key)[:n]:
            keep[b, p] = 0
    return keep


def test_select_keep_hand_example():
    from oracle.compaction import select_keep
    # scores of one sequence; filter the 3 lowest: -2.0 (pos 4), then the two
    # 0.5s -- equal, so the lower position (1) goes before (3) -- nothing else
    s = np.array([[1.0, 0.5, 7.0, 0.5, -2.0, 0.5]], np.float32)
    assert select_keep(s, 3).tolist() == [[1, 0, 1, 0, 0, 1]]
    assert select_keep(s, 0).tolist() == [[1] * 6]
    assert select_keep(s, 6).tolist() == [[0] * 6]


def test_select_keep_brute_force():
    from oracle.compaction import select_keep
    rng = np.random.default_rng(5)
    s = rng.integers(-3, 4, size=(3, 40)).astype(np.float32)      # many ties
    s[0, 5] = np.nan
    s[1, 7] = -0.0
    s[1, 8] = 0.0
    s[2, :3] = np.inf
    for n in (0, 1, 13, 39, 40):
        assert np.array_equal(select_keep(s, n), _brute_select(s, n))
    # matches the generator's Gumbel rule on the same scores
    g = np.random.Generator(np.random.PCG64(123)).gumbel(size=(2, 64))
    import workloads
    want = workloads.gumbel_keep_mask(2, 64, 0.4, 123)
    assert np.array_equal(select_keep(g.astype(np.float32), workloads.n_filtered(64, 0.4)), want)
