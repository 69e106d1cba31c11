"""GPU failure detection without a GPU fault: a bounded in-kernel wait that
runs out, and a kept index outside its buffer, both come back through
collider_check as status codes, and the device stays usable afterwards."""
import numpy as np
import pytest
import torch

import workloads
from oracle import compaction

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
cl = gu.cl


def _compaction_still_works():
    keep = workloads.gumbel_keep_mask(3, 500, 0.4, seed=5)
    idx, cu, nk = gu.compact(keep)
    cl.collider_check()
    ridx, rcu, rnk = compaction.compact(keep)
    assert int(nk.item()) == rnk
    assert np.array_equal(idx[:rnk].cpu().numpy(), ridx)
    assert np.array_equal(cu.cpu().numpy(), rcu)


def test_wait_that_runs_out_is_reported_and_cleared():
    cl.collider_check()                      # nothing pending
    cl.collider_selftest_wait_timeout()
    with pytest.raises(cl.ColliderError) as e:
        cl.collider_check()
    assert e.value.status == cl.ERR_TIMEOUT
    assert "site 999" in str(e.value)
    cl.collider_check()                      # the status word was cleared
    _compaction_still_works()


def test_kept_index_outside_the_buffer_is_skipped_and_reported():
    M, row = 64, 256
    src = torch.arange(M * row // 2, dtype=torch.int16, device=gu.DEV).view(M, row // 2)
    dst = torch.full((M, row // 2), -7, dtype=torch.int16, device=gu.DEV)
    idx = torch.tensor([3, 5, M + 5, 9], dtype=torch.int32, device=gu.DEV)
    nk = torch.tensor([4], dtype=torch.int32, device=gu.DEV)
    cl.collider_gather_rows(src, row, dst, row, row, M, idx, nk)
    with pytest.raises(cl.ColliderError) as e:
        cl.collider_check()
    assert e.value.status == cl.ERR_INVALID_ARG
    assert "index outside its buffer" in str(e.value)
    # the rows with valid indices were gathered; the bad one was left alone
    got = dst.cpu().numpy()
    ref = src.cpu().numpy()
    assert np.array_equal(got[0], ref[3]) and np.array_equal(got[1], ref[5]) and np.array_equal(got[3], ref[9])
    assert np.all(got[2] == -7)
    cl.collider_check()
    _compaction_still_works()
