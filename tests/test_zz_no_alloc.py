"""gs_sort_pairs_noalloc, the sort for callers that cannot allocate device
memory (and so cannot pass a workspace), must give exactly what the
workspace-taking gs_sort_pairs gives.  Two calls in a row, with different
sizes and bit ranges, check that the shared scratch array's leftovers from
one call do not leak into the next.  This file is collected last."""

import ctypes as ct

import numpy as np
import pytest
import torch

from tile_gaussian_splat_gb300 import binding as gs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _pairs(seed, n, distinct):
    rng = np.random.default_rng(seed)
    pool = rng.integers(0, 2**63, distinct, dtype=np.uint64) * np.uint64(2) + \
        rng.integers(0, 2, distinct, dtype=np.uint64)
    keys = rng.choice(pool, n).astype(np.uint64)
    return (torch.from_numpy(keys.view(np.int64).copy()).to(DEV),
            torch.from_numpy(np.arange(n, dtype=np.int32)).to(DEV))


def test_noalloc_sort_equals_workspace_sort_twice():
    lib = gs.lib()
    # pass counts 8, 2 (even: the result ends in the caller's arrays), 3 at
    # the largest n (odd: it ends in the library's alternate buffers and is
    # copied back, with the array's capacity fully used) and 5
    cases = [(1, 600_001, 5000, 0, 64), (2, 250_000, 300, 32, 47),
             (3, gs.SORT_NOALLOC_MAX_PAIRS, 7000, 0, 24), (4, 1000, 50, 8, 48)]
    for seed, n, distinct, b0, b1 in cases:
        k_ref, v_ref = _pairs(seed, n, distinct)
        k, v = k_ref.clone(), v_ref.clone()
        gs.gs_sort_pairs(k_ref, v_ref, b0, b1)
        st = gs.new_status(DEV)
        rc = lib.gs_sort_pairs_noalloc(k.data_ptr(), v.data_ptr(), n, b0, b1, st.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        assert int(st.item()) == 0
        assert torch.equal(k, k_ref) and torch.equal(v, v_ref)


def test_noalloc_sort_rejects_oversize():
    n = gs.SORT_NOALLOC_MAX_PAIRS + 1
    k = torch.zeros(n, dtype=torch.int64, device=DEV)
    v = torch.zeros(n, dtype=torch.int32, device=DEV)
    rc = gs.lib().gs_sort_pairs_noalloc(k.data_ptr(), v.data_ptr(), n, 0, 64, None,
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == 2  # GS_ERR_CAPACITY
