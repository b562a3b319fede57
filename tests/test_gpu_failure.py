"""The failure path of the bounded inter-block waits, made to happen on
purpose without a fault: a sorting pass whose first look-back word is never
published (its block ticket starts past 0) and whose waits give up after a
few thousand polls must report GS_ERR_TIMEOUT in the status word, return,
and leave the context usable (the pages' sort, gsplat 1.0.0, intersections.c,
gs_radix_sort_without_gvl, returns an error instead of aborting)."""

import time

import numpy as np
import pytest
import torch

from tile_gaussian_splat_gb300 import binding as gs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.mark.parametrize("n,ticket_start", [(5000, 1), (20000, 3), (300, 2)])
def test_lookback_wait_runs_out_and_reports_timeout(n, ticket_start):
    rng = np.random.default_rng(n)
    keys = torch.from_numpy(rng.integers(0, 2**62, n, dtype=np.int64)).to(DEV)
    vals = torch.arange(n, dtype=torch.int32, device=DEV)
    st = gs.new_status(DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    gs.gs_debug_sort_wait_timeout(keys, vals, ticket_start, 4096, st)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) == 5  # GS_ERR_TIMEOUT
    assert elapsed < 5.0
    # the context still works: a normal sort right after is exact
    k = torch.from_numpy(rng.integers(0, 2**62, 70001, dtype=np.int64)).to(DEV)
    v = torch.arange(70001, dtype=torch.int32, device=DEV)
    ref = np.argsort(k.cpu().numpy(), kind="stable")
    st2 = gs.new_status(DEV)
    gs.gs_sort_pairs(k, v, 0, 64, d_status=st2)
    gs.check_status(st2)
    np.testing.assert_array_equal(v.cpu().numpy(), ref)
