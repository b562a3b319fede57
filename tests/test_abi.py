"""The C ABI library loads on a CPU-only machine and exports every symbol
include/gs_splat.h declares; host-side argument checks answer without a GPU
(they return before any CUDA call)."""

import ctypes as ct
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from tile_gaussian_splat_gb300 import build, binding
    build.build()
    return binding.lib()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(gs_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    from tile_gaussian_splat_gb300 import binding
    assert set(binding.SIGNATURES) == set(names)


def test_host_only_entry_points(lib):
    assert lib.gs_version() == 100
    assert lib.gs_status_string(3) == b"intersection key is outside the tile grid"
    assert lib.gs_status_string(99) == b"unknown status"
    for (w, h), b in [((1, 1), 0), ((4, 4), 4), ((120, 68), 13), ((240, 135), 15)]:
        assert lib.gs_tile_bits(w, h) == b
    q = lib.gs_isect_workspace_size(4, 1000, 120, 68, 0, 1)
    e = lib.gs_isect_workspace_size(4, 1000, 120, 68, 100000, 1)
    assert 0 < q < e
    assert lib.gs_sort_workspace_size(1000) > 12 * 1000


def test_argument_errors_without_gpu(lib):
    P = ct.c_void_p
    # C = 0, tile_size = 0, too many key bits: rejected on the host
    assert lib.gs_isect_tiles(None, None, 0, None, 0, 10, 16, 4, 4, 1, None, None, None, None,
                              0, None, 0, None, None) == 1
    assert lib.gs_isect_tiles(P(8), P(8), 0, P(8), 1, 10, 0, 4, 4, 1, None, None, None, None, 0,
                              None, 0, None, None) == 1
    assert lib.gs_isect_tiles(P(8), P(8), 0, P(8), 65537, 1, 16, 256, 256, 1, None, None, None,
                              None, 0, None, 0, None, None) == 1
    # query without a host total pointer
    assert lib.gs_isect_tiles(P(8), P(8), 0, P(8), 1, 10, 16, 4, 4, 1, None, None, None, None,
                              0, None, 0, None, None) == 1
    # query with no workspace
    total = ct.c_int64()
    assert lib.gs_isect_tiles(P(8), P(8), 0, P(8), 1, 10, 16, 4, 4, 1, None, ct.byref(total),
                              None, None, 0, None, 0, None, None) == 4
    assert lib.gs_tile_offsets(None, 5, 1, 4, 4, P(8), None, None) == 1
    # channel counts outside 1..GS_MAX_CHANNELS (1024) and tile sizes other than 16
    for ch, ts in ((0, 16), (1025, 16), (3, 8)):
        assert lib.gs_rasterize_fwd(P(8), P(8), P(8), P(8), None, None, 1, 10, ch, 64, 64, ts,
                                    P(8), P(8), 10, ct.c_float(0.1), ct.c_float(0.1), P(8), P(8),
                                    P(8), None, None, None, None) == 1
    assert lib.gs_sort_pairs(None, None, 5, 0, 64, None, 0, None, None) == 1
    assert lib.gs_sort_pairs(P(8), P(8), 5, 0, 65, None, 0, None, None) == 1
    assert lib.gs_sort_pairs(P(8), P(8), 5, 0, 64, None, 0, None, None) == 4


def test_timeout_hook_argument_errors_without_gpu(lib):
    P = ct.c_void_p
    call = lambda n, t, w, ws=P(8), nb=1 << 40, st=P(8): lib.gs_debug_sort_wait_timeout(
        P(8), P(8), n, t, w, ws, nb, st, None)
    assert call(0, 1, 10) == 1             # n = 0
    assert call(100, 0, 10) == 1           # ticket_start must be >= 1
    assert call(100, 65, 10) == 1          # at most 64
    assert call(100, 1, 0) == 1            # wait_polls >= 1
    assert call(100, 1, (1 << 20) + 1) == 1
    assert call(100, 1, 10, st=None) == 1  # the status word is required
    assert call(100, 1, 10, ws=None) == 4  # workspace missing
    assert call(100, 2, 10, nb=lib.gs_sort_workspace_size(100 + 2 * 2048) - 1) == 4
