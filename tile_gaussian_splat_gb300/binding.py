"""Python binding of libgs_splat_gb300 (include/gs_splat.h).

Argument marshalling only: every function hands torch CUDA tensors' device
pointers and the current stream to the C entry point of the same name, and
allocates what the C call needs (outputs and workspace) with torch.  Every
step of the path runs in the library's kernels.  There is no CPU fallback:
if the library is missing or no GPU is present, calls raise.
"""

from __future__ import annotations

import contextlib
import ctypes as ct
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgs_splat_gb300.so")
LIB_DEBUG_PATH = os.path.join(_HERE, "libgs_splat_gb300_debug.so")

GS_OK = 0
STATUS_NAMES = {
    0: "GS_OK", 1: "GS_ERR_INVALID_ARG", 2: "GS_ERR_CAPACITY", 3: "GS_ERR_KEY_OUT_OF_GRID",
    4: "GS_ERR_WORKSPACE", 5: "GS_ERR_TIMEOUT", 6: "GS_ERR_CUDA", 7: "GS_ERR_UNSORTED",
    8: "GS_ERR_COUNT_MISMATCH", 9: "GS_ERR_OUT_OF_BOUNDS",
}

# exported symbol -> (restype, argtypes); mirrors include/gs_splat.h
P, I32, I64, F32, SZ = ct.c_void_p, ct.c_int, ct.c_int64, ct.c_float, ct.c_size_t
SIGNATURES = {
    "gs_version": (I32, []),
    "gs_status_string": (ct.c_char_p, [I32]),
    "gs_tile_bits": (I32, [I32, I32]),
    "gs_isect_workspace_size": (SZ, [I32, I32, I32, I32, I64, I32]),
    "gs_isect_tiles": (I32, [P, P, I32, P, I32, I32, I32, I32, I32, I32, P, P, P, P, I64, P, SZ,
                             P, P]),
    "gs_tile_offsets": (I32, [P, I64, I32, I32, I32, P, P, P]),
    "gs_rasterize_fwd": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P, I64, F32,
                               F32, P, P, P, P, P, P, P]),
    "gs_rasterize_bwd": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P, I64, F32,
                               P, P, P, P, P, P, P, P, P, P, P, P, P]),
    "gs_project": (I32, [P, P, P, P, I32, I32, I32, I32, F32, F32, F32, F32, I32, P, P, P, P, P,
                         P, P, P]),
    "gs_bin_splats": (I32, [P, P, I32, P, I32, I32, I32, I32, I32, I32, P, P, P, P]),
    "gs_rasterize_fwd_bins": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P, I32,
                                    F32, F32, P, P, P, P, P, P, P]),
    "gs_rasterize_bwd_bins": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P, I32,
                                    F32, P, P, P, P, P, P, P, P, P, P, P, P, P]),
    "gs_sort_workspace_size": (SZ, [I64]),
    "gs_sort_pairs": (I32, [P, P, I64, I32, I32, P, SZ, P, P]),
    "gs_sort_pairs_noalloc": (I32, [P, P, I64, I32, I32, P, P]),
    "gs_debug_sort_wait_timeout": (I32, [P, P, I64, I32, I32, P, SZ, P, P]),
    "gs_peak_probe": (I32, [I32, I32, I32, P, P, P]),
    "gs_rasterize_fwd_steps": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P, I64,
                                     F32, F32, I32, P, P, P, P, P, P, P, P]),
    "gs_rasterize_bwd_steps": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P, I64,
                                     F32, P, P, I32, P, P, P, P, P, P, P, P, P, P, P, P, P]),
}


class GsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_status_text(code)})")


_lib = None


def _load(path):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; "
            "g.build()'` (the CUDA library has no CPU fallback)")
    L = ct.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """Opens the library (once).  Raises if it was not built."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


@contextlib.contextmanager
def library(path):
    """Routes this module's calls to another build of the library -- the
    range-checking build, LIB_DEBUG_PATH -- while the block runs."""
    global _lib
    saved = _lib
    _lib = _load(path)
    try:
        yield _lib
    finally:
        _lib = saved


def _status_text(code):
    try:
        return lib().gs_status_string(code).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(code, where):
    if code != GS_OK:
        raise GsError(code, where)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr() or None


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(d_status: torch.Tensor, where: str = "device"):
    """Reads a device status word (synchronises) and raises on an error."""
    code = int(d_status.item())
    _check(code, where)


def gs_tile_bits(tile_width: int, tile_height: int) -> int:
    return int(lib().gs_tile_bits(tile_width, tile_height))


def gs_isect_workspace_size(C, N, tile_width, tile_height, n_isects, sort=True) -> int:
    return int(lib().gs_isect_workspace_size(C, N, tile_width, tile_height, n_isects, int(sort)))


def gs_isect_tiles(means2d, radii, depths, tile_size, tile_width, tile_height, sort=True,
                   d_status=None, workspace=None, stream=None):
    """Both calls of the C entry point: the size query, then the emission.
    Returns (tiles_per_gauss (C,N) int32, keys (I,) int64 holding the uint64
    bits, flatten_ids (I,) int32)."""
    C, N = means2d.shape[:2]
    dev = means2d.device
    ell = int(radii.dim() == 3)
    tpg = _empty((C, N), torch.int32, dev)
    s = _stream(stream)
    q_bytes = gs_isect_workspace_size(C, N, tile_width, tile_height, 0, sort)
    ws = workspace if workspace is not None and workspace.numel() >= q_bytes else \
        _empty(q_bytes, torch.uint8, dev)
    total = ct.c_int64(0)
    _check(lib().gs_isect_tiles(_ptr(means2d), _ptr(radii), ell, _ptr(depths), C, N, tile_size,
                                tile_width, tile_height, int(sort), _ptr(tpg), ct.byref(total),
                                None, None, 0, _ptr(ws), ws.numel(), _ptr(d_status), s),
           "gs_isect_tiles (size query)")
    I = int(total.value)
    keys = _empty(I, torch.int64, dev)
    ids = _empty(I, torch.int32, dev)
    if I == 0:
        return tpg, keys, ids
    e_bytes = gs_isect_workspace_size(C, N, tile_width, tile_height, I, sort)
    if ws.numel() < e_bytes:
        ws = _empty(e_bytes, torch.uint8, dev)
    _check(lib().gs_isect_tiles(_ptr(means2d), _ptr(radii), ell, _ptr(depths), C, N, tile_size,
                                tile_width, tile_height, int(sort), None, None, _ptr(keys),
                                _ptr(ids), I, _ptr(ws), ws.numel(), _ptr(d_status), s),
           "gs_isect_tiles")
    return tpg, keys, ids


def gs_tile_offsets(keys, C, tile_width, tile_height, d_status=None, out=None, stream=None):
    """offsets (C, tile_height, tile_width) int32 from sorted keys."""
    offsets = out if out is not None else _empty((C, tile_height, tile_width), torch.int32,
                                                 keys.device)
    _check(lib().gs_tile_offsets(_ptr(keys), keys.numel(), C, tile_width, tile_height,
                                 _ptr(offsets), _ptr(d_status), _stream(stream)),
           "gs_tile_offsets")
    return offsets


def gs_project(means, covars, viewmats, intrinsics, width, height, eps2d=0.3, near_plane=0.01,
               far_plane=1e10, radius_clip=0.0, compensation=False, orthographic=False,
               radii_float=False, d_status=None, out=None, stream=None):
    """EWA projection.  means (N,3), covars (N,3,3), viewmats (C,4,4),
    intrinsics (C,3,3), float32 CUDA tensors.  Returns dict(radii int32
    (C,N,2), means2d (C,N,2), depths (C,N), conics (C,N,3), compensations
    (C,N) or None, radii_float (C,N,2) or None: the radii as gs_isect_tiles
    takes them)."""
    N = means.shape[0]
    C = viewmats.shape[0]
    dev = means.device
    if out is None:
        out = dict(radii=_empty((C, N, 2), torch.int32, dev),
                   means2d=_empty((C, N, 2), torch.float32, dev),
                   depths=_empty((C, N), torch.float32, dev),
                   conics=_empty((C, N, 3), torch.float32, dev),
                   compensations=_empty((C, N), torch.float32, dev) if compensation else None,
                   radii_float=_empty((C, N, 2), torch.float32, dev) if radii_float else None)
    _check(lib().gs_project(
        _ptr(means), _ptr(covars), _ptr(viewmats), _ptr(intrinsics), C, N, int(width),
        int(height), float(eps2d), float(near_plane), float(far_plane), float(radius_clip),
        int(bool(orthographic)), _ptr(out["radii"]), _ptr(out["means2d"]), _ptr(out["depths"]),
        _ptr(out["conics"]), _ptr(out["compensations"]), _ptr(out["radii_float"]),
        _ptr(d_status), _stream(stream)), "gs_project")
    return out


def gs_bin_splats(means2d, radii, depths, tile_size, tile_width, tile_height, capacity,
                  d_status=None, out=None, stream=None):
    """Returns (bins int32 (C, TH, TW, capacity) with -1 after each bin's
    splats, bin_counts int32 (C, TH, TW))."""
    C, N = means2d.shape[:2]
    dev = means2d.device
    if out is None:
        out = (_empty((C, tile_height, tile_width, capacity), torch.int32, dev),
               _empty((C, tile_height, tile_width), torch.int32, dev))
    bins, counts = out
    _check(lib().gs_bin_splats(
        _ptr(means2d), _ptr(radii), int(radii.dim() == 3), _ptr(depths), C, N, tile_size,
        tile_width, tile_height, int(capacity), _ptr(bins), _ptr(counts), _ptr(d_status),
        _stream(stream)), "gs_bin_splats")
    return bins, counts


def gs_rasterize_fwd(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                     tile_size, offsets, flatten_ids, alpha_cutoff, transmittance_threshold,
                     d_status=None, out=None, pair_counts=None, trace=None, stream=None):
    """Returns (render_colors (C,H,W,ch), render_alphas (C,H,W,1), last_ids (C,H,W)).
    pair_counts: optional int32 (C,H,W,3) tensor that receives per pixel the
    entries evaluated, the entries composited and the entries evaluated up
    to the last composited one.  trace: optional int32 (n_isects, 8) tensor
    that receives the per-entry composite masks for gs_rasterize_bwd."""
    C, N = means2d.shape[:2]
    ch = colors.shape[-1]
    dev = means2d.device
    if out is None:
        out = (_empty((C, height, width, ch), torch.float32, dev),
               _empty((C, height, width, 1), torch.float32, dev),
               _empty((C, height, width), torch.int32, dev))
    rgb, alpha, last = out
    _check(lib().gs_rasterize_fwd(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, _ptr(offsets), _ptr(flatten_ids),
        flatten_ids.numel(), float(alpha_cutoff), float(transmittance_threshold), _ptr(rgb),
        _ptr(alpha), _ptr(last), _ptr(pair_counts), _ptr(trace), _ptr(d_status),
        _stream(stream)), "gs_rasterize_fwd")
    return rgb, alpha, last


def gs_rasterize_bwd(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                     tile_size, offsets, flatten_ids, alpha_cutoff, render_alphas, last_ids,
                     grad_render_colors, grad_render_alphas, want_grad_backgrounds=None,
                     absgrad=False, d_status=None, out=None, trace=None, stream=None):
    """Returns dict(grad_means2d, grad_conics, grad_colors, grad_opacities,
    grad_backgrounds (or None), grad_means2d_abs (or None)).  trace: the mask
    table the forward wrote for the same inputs (optional, faster)."""
    C, N = means2d.shape[:2]
    ch = colors.shape[-1]
    dev = means2d.device
    if want_grad_backgrounds is None:
        want_grad_backgrounds = backgrounds is not None
    if out is None:
        out = dict(grad_means2d=_empty((C, N, 2), torch.float32, dev),
                   grad_conics=_empty((C, N, 3), torch.float32, dev),
                   grad_colors=_empty((C, N, ch), torch.float32, dev),
                   grad_opacities=_empty((C, N), torch.float32, dev),
                   grad_backgrounds=_empty((C, ch), torch.float32, dev)
                   if want_grad_backgrounds else None,
                   grad_means2d_abs=_empty((C, N, 2), torch.float32, dev) if absgrad else None)
    _check(lib().gs_rasterize_bwd(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, _ptr(offsets), _ptr(flatten_ids),
        flatten_ids.numel(), float(alpha_cutoff), _ptr(render_alphas), _ptr(last_ids),
        _ptr(grad_render_colors), _ptr(grad_render_alphas), _ptr(out["grad_means2d"]),
        _ptr(out["grad_conics"]), _ptr(out["grad_colors"]), _ptr(out["grad_opacities"]),
        _ptr(out["grad_backgrounds"]), _ptr(out["grad_means2d_abs"]), _ptr(trace),
        _ptr(d_status), _stream(stream)), "gs_rasterize_bwd")
    return out


def gs_sort_pairs(keys, values, begin_bit=0, end_bit=64, d_status=None, workspace=None,
                  stream=None):
    """Stable in-place sort of (keys int64 holding uint64 bits, values int32)
    by key bits [begin_bit, end_bit)."""
    n = keys.numel()
    need = int(lib().gs_sort_workspace_size(n))
    ws = workspace if workspace is not None and workspace.numel() >= need else \
        _empty(max(need, 1), torch.uint8, keys.device)
    _check(lib().gs_sort_pairs(_ptr(keys), _ptr(values), n, begin_bit, end_bit, _ptr(ws),
                               ws.numel(), _ptr(d_status), _stream(stream)), "gs_sort_pairs")
    return keys, values


SORT_NOALLOC_MAX_PAIRS = 1 << 20


def gs_sort_pairs_noalloc(keys, values, begin_bit=0, end_bit=64, d_status=None, stream=None):
    """gs_sort_pairs without a workspace: the library's own fixed scratch
    array is used (n <= SORT_NOALLOC_MAX_PAIRS; calls on one device must not
    overlap on the GPU)."""
    _check(lib().gs_sort_pairs_noalloc(_ptr(keys), _ptr(values), keys.numel(), begin_bit,
                                       end_bit, _ptr(d_status), _stream(stream)),
           "gs_sort_pairs_noalloc")
    return keys, values


def gs_rasterize_fwd_bins(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                          tile_size, bins, bin_counts, alpha_cutoff, transmittance_threshold,
                          d_status=None, out=None, pair_counts=None, trace=None, stream=None):
    """gs_rasterize_fwd over bin lists (bins (C, TH, TW, M), bin_counts).
    last_ids and trace rows are positions in bins."""
    C, N = means2d.shape[:2]
    ch = colors.shape[-1]
    dev = means2d.device
    if out is None:
        out = (_empty((C, height, width, ch), torch.float32, dev),
               _empty((C, height, width, 1), torch.float32, dev),
               _empty((C, height, width), torch.int32, dev))
    rgb, alpha, last = out
    _check(lib().gs_rasterize_fwd_bins(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, _ptr(bins), _ptr(bin_counts),
        bins.shape[-1], float(alpha_cutoff), float(transmittance_threshold), _ptr(rgb),
        _ptr(alpha), _ptr(last), _ptr(pair_counts), _ptr(trace), _ptr(d_status),
        _stream(stream)), "gs_rasterize_fwd_bins")
    return rgb, alpha, last


def gs_rasterize_bwd_bins(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                          tile_size, bins, bin_counts, alpha_cutoff, render_alphas, last_ids,
                          grad_render_colors, grad_render_alphas, want_grad_backgrounds=None,
                          absgrad=False, d_status=None, out=None, trace=None, stream=None):
    """gs_rasterize_bwd over bin lists; same outputs as gs_rasterize_bwd."""
    C, N = means2d.shape[:2]
    ch = colors.shape[-1]
    dev = means2d.device
    if want_grad_backgrounds is None:
        want_grad_backgrounds = backgrounds is not None
    if out is None:
        out = dict(grad_means2d=_empty((C, N, 2), torch.float32, dev),
                   grad_conics=_empty((C, N, 3), torch.float32, dev),
                   grad_colors=_empty((C, N, ch), torch.float32, dev),
                   grad_opacities=_empty((C, N), torch.float32, dev),
                   grad_backgrounds=_empty((C, ch), torch.float32, dev)
                   if want_grad_backgrounds else None,
                   grad_means2d_abs=_empty((C, N, 2), torch.float32, dev) if absgrad else None)
    _check(lib().gs_rasterize_bwd_bins(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, _ptr(bins), _ptr(bin_counts),
        bins.shape[-1], float(alpha_cutoff), _ptr(render_alphas), _ptr(last_ids),
        _ptr(grad_render_colors), _ptr(grad_render_alphas), _ptr(out["grad_means2d"]),
        _ptr(out["grad_conics"]), _ptr(out["grad_colors"]), _ptr(out["grad_opacities"]),
        _ptr(out["grad_backgrounds"]), _ptr(out["grad_means2d_abs"]), _ptr(trace),
        _ptr(d_status), _stream(stream)), "gs_rasterize_bwd_bins")
    return out


def gs_debug_sort_wait_timeout(keys, values, ticket_start, wait_polls, d_status, stream=None):
    """Test hook of the timeout path (see the header): one sorting pass whose
    first look-back word is never published and whose waits poll at most
    wait_polls times.  keys int64 (n), values int32 (n) are overwritten with
    unspecified values; d_status receives GS_ERR_TIMEOUT."""
    n = keys.numel()
    ws = _empty(lib().gs_sort_workspace_size(n + ticket_start * 2048), torch.uint8, keys.device)
    _check(lib().gs_debug_sort_wait_timeout(_ptr(keys), _ptr(values), n, ticket_start,
                                            wait_polls, _ptr(ws), ws.numel(), _ptr(d_status),
                                            _stream(stream)), "gs_debug_sort_wait_timeout")
    return ws


def gs_peak_probe(kind, iters, blocks, out, stream=None):
    """Enqueues the throughput probe (kind 0 FMA, 1 packed FMA, 2 ex2) into
    out (float32, blocks * 256); returns the number of operations."""
    ops = ct.c_int64(0)
    _check(lib().gs_peak_probe(kind, iters, blocks, _ptr(out), ct.byref(ops), _stream(stream)),
           "gs_peak_probe")
    return int(ops.value)


def gs_rasterize_fwd_steps(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                           tile_size, offsets, flatten_ids, alpha_cutoff,
                           transmittance_threshold, max_steps, d_status=None, stream=None):
    """gs_rasterize_fwd that also records the per-pixel step trace.  Returns
    (render_colors, render_alphas, last_ids, (step_pos, step_T, step_count))
    with step_pos int32 / step_T float32 (max_steps, C, H, W) and step_count
    int32 (C, H, W)."""
    C, N = means2d.shape[0], means2d.shape[1]
    ch = colors.shape[-1]
    dev = means2d.device
    rgb = _empty((C, height, width, ch), torch.float32, dev)
    alpha = _empty((C, height, width, 1), torch.float32, dev)
    last = _empty((C, height, width), torch.int32, dev)
    pos = _empty((max_steps, C, height, width), torch.int32, dev)
    tb = _empty((max_steps, C, height, width), torch.float32, dev)
    cnt = _empty((C, height, width), torch.int32, dev)
    _check(lib().gs_rasterize_fwd_steps(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, _ptr(offsets), _ptr(flatten_ids),
        flatten_ids.numel(), alpha_cutoff, transmittance_threshold, max_steps, _ptr(rgb),
        _ptr(alpha), _ptr(last), _ptr(pos), _ptr(tb), _ptr(cnt), _ptr(d_status),
        _stream(stream)), "gs_rasterize_fwd_steps")
    return rgb, alpha, last, (pos, tb, cnt)


def gs_rasterize_bwd_steps(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                           tile_size, offsets, flatten_ids, alpha_cutoff, render_alphas,
                           last_ids, steps, grad_render_colors, grad_render_alphas,
                           absgrad=False, d_status=None, out=None, stream=None):
    """The backward over a step trace `steps` = (step_pos, step_T, step_count)
    from gs_rasterize_fwd_steps.  Returns the gradients as gs_rasterize_bwd."""
    C, N = means2d.shape[0], means2d.shape[1]
    ch = colors.shape[-1]
    dev = means2d.device
    pos, tb, cnt = steps
    if out is None:
        out = dict(grad_means2d=_empty((C, N, 2), torch.float32, dev),
                   grad_conics=_empty((C, N, 3), torch.float32, dev),
                   grad_colors=_empty((C, N, ch), torch.float32, dev),
                   grad_opacities=_empty((C, N), torch.float32, dev),
                   grad_backgrounds=None if backgrounds is None else
                   _empty((C, ch), torch.float32, dev),
                   grad_means2d_abs=_empty((C, N, 2), torch.float32, dev) if absgrad else None)
    _check(lib().gs_rasterize_bwd_steps(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, _ptr(offsets), _ptr(flatten_ids),
        flatten_ids.numel(), alpha_cutoff, _ptr(render_alphas), _ptr(last_ids), pos.shape[0],
        _ptr(pos), _ptr(tb), _ptr(cnt), _ptr(grad_render_colors), _ptr(grad_render_alphas),
        _ptr(out["grad_means2d"]), _ptr(out["grad_conics"]), _ptr(out["grad_colors"]),
        _ptr(out["grad_opacities"]), _ptr(out["grad_backgrounds"]),
        _ptr(out["grad_means2d_abs"]), _ptr(d_status), _stream(stream)),
        "gs_rasterize_bwd_steps")
    return out
