"""A C program -- no Python, no PyTorch -- drives one training step through
the C ABI (size query, emission, tile offsets, forward with the trace,
backward) on a scene the test writes to files.  Its outputs equal those of
the same calls made through the binding: bit for bit for the indexing and
forward outputs, the gradients up to the order of float atomics."""

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from gpu_util import DEV, to_dev
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "gs_splat.h"

static const char* dir;

static void* dev_alloc(size_t bytes) {
    void* p = NULL;
    if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) { fprintf(stderr, "cudaMalloc\n"); exit(2); }
    cudaMemset(p, 0, bytes ? bytes : 16);
    return p;
}

static void* load(const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s.bin", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) { fprintf(stderr, "open %s\n", path); exit(2); }
    void* h = malloc(bytes);
    if (fread(h, 1, bytes, f) != bytes) { fprintf(stderr, "read %s\n", path); exit(2); }
    fclose(f);
    void* d = dev_alloc(bytes);
    cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice);
    free(h);
    return d;
}

static void save(const char* name, const void* d, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/out_%s.bin", dir, name);
    void* h = malloc(bytes ? bytes : 1);
    cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost);
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(h, 1, bytes, f) != bytes) { fprintf(stderr, "write %s\n", path); exit(2); }
    fclose(f);
    free(h);
}

#define CALL(x) do { int rc_ = (x); if (rc_ != GS_OK) { \
    fprintf(stderr, "%s: %s\n", #x, gs_status_string(rc_)); return 3; } } while (0)

int main(int argc, char** argv) {
    if (argc != 6) return 1;
    dir = argv[1];
    const int C = atoi(argv[2]), N = atoi(argv[3]), W = atoi(argv[4]), H = atoi(argv[5]);
    const int TW = (W + 15) / 16, TH = (H + 15) / 16;
    const size_t CN = (size_t)C * N, P = (size_t)C * H * W;
    float* means2d = load("means2d", CN * 2 * 4);
    float* radii = load("radii", CN * 2 * 4);
    float* depths = load("depths", CN * 4);
    float* conics = load("conics", CN * 3 * 4);
    float* colors = load("colors", CN * 3 * 4);
    float* opacities = load("opacities", CN * 4);
    float* g_rgb = load("grad_render_colors", P * 3 * 4);
    float* g_a = load("grad_render_alphas", P * 4);
    int32_t* status = dev_alloc(4);
    int32_t* tpg = dev_alloc(CN * 4);

    size_t ws = gs_isect_workspace_size(C, N, TW, TH, 0, 1);
    void* work = dev_alloc(ws);
    int64_t I = 0;
    CALL(gs_isect_tiles(means2d, radii, 1, depths, C, N, 16, TW, TH, 1, tpg, &I, NULL, NULL,
                        0, work, ws, status, NULL));
    cudaFree(work);
    ws = gs_isect_workspace_size(C, N, TW, TH, I, 1);
    work = dev_alloc(ws);
    uint64_t* keys = dev_alloc((size_t)I * 8);
    int32_t* ids = dev_alloc((size_t)I * 4);
    CALL(gs_isect_tiles(means2d, radii, 1, depths, C, N, 16, TW, TH, 1, tpg, NULL, keys, ids,
                        I, work, ws, status, NULL));
    int32_t* offsets = dev_alloc((size_t)C * TH * TW * 4);
    CALL(gs_tile_offsets(keys, I, C, TW, TH, offsets, status, NULL));
    float* rgb = dev_alloc(P * 3 * 4);
    float* alpha = dev_alloc(P * 4);
    int32_t* last = dev_alloc(P * 4);
    uint32_t* trace = dev_alloc((size_t)I * 8 * 4);
    CALL(gs_rasterize_fwd(means2d, conics, colors, opacities, NULL, NULL, C, N, 3, W, H, 16,
                          offsets, ids, I, 1.0f / 255.0f, 1e-4f, rgb, alpha, last, NULL, trace,
                          status, NULL));
    float* gm = dev_alloc(CN * 2 * 4);
    float* gc = dev_alloc(CN * 3 * 4);
    float* gcol = dev_alloc(CN * 3 * 4);
    float* gop = dev_alloc(CN * 4);
    CALL(gs_rasterize_bwd(means2d, conics, colors, opacities, NULL, NULL, C, N, 3, W, H, 16,
                          offsets, ids, I, 1.0f / 255.0f, alpha, last, g_rgb, g_a, gm, gc, gcol,
                          gop, NULL, NULL, trace, status, NULL));
    if (cudaDeviceSynchronize() != cudaSuccess) { fprintf(stderr, "sync\n"); return 4; }
    int32_t st = 0;
    cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost);
    save("tiles_per_gauss", tpg, CN * 4);
    save("keys", keys, (size_t)I * 8);
    save("flatten_ids", ids, (size_t)I * 4);
    save("offsets", offsets, (size_t)C * TH * TW * 4);
    save("render_colors", rgb, P * 3 * 4);
    save("render_alphas", alpha, P * 4);
    save("last_ids", last, P * 4);
    save("grad_means2d", gm, CN * 2 * 4);
    save("grad_conics", gc, CN * 3 * 4);
    save("grad_colors", gcol, CN * 3 * 4);
    save("grad_opacities", gop, CN * 4);
    printf("%lld %d\n", (long long)I, st);
    return st == GS_OK ? 0 : 5;
}
"""


def _build(tmp):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = os.path.join(tmp, "step.c")
    exe = os.path.join(tmp, "step")
    with open(src, "w") as f:
        f.write(C_SOURCE)
    libdir = os.path.join(ROOT, "tile_gaussian_splat_gb300")
    r = subprocess.run([nvcc, "-O1", src, "-o", exe, "-I", os.path.join(ROOT, "include"),
                        "-L", libdir, "-lgs_splat_gb300", "-Xlinker", f"-rpath={libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return exe


def test_c_program_runs_a_training_step(tmp_path):
    s = scenes.random_small(21, C=2, N=3000, W=150, H=90, sigma=(0.5, 10.0))
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, seed=4)
    tmp = str(tmp_path)
    inputs = {"means2d": s.means2d, "radii": s.radii, "depths": s.depths, "conics": s.conics,
              "colors": s.colors, "opacities": s.opacities, "grad_render_colors": g_rgb,
              "grad_render_alphas": g_a}
    for k, v in inputs.items():
        np.ascontiguousarray(v, dtype=np.float32).tofile(os.path.join(tmp, k + ".bin"))
    exe = _build(tmp)
    r = subprocess.run([exe, tmp, str(s.C), str(s.N), str(s.width), str(s.height)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.stdout, r.stderr)
    I = int(r.stdout.split()[0])

    def out(name, dtype, shape):
        return np.fromfile(os.path.join(tmp, f"out_{name}.bin"), dtype=dtype).reshape(shape)

    # the same calls through the binding
    d = {k: to_dev(v) for k, v in inputs.items()}
    st = gs.new_status(DEV)
    tpg, keys, ids = gs.gs_isect_tiles(d["means2d"], d["radii"], d["depths"], 16,
                                       s.tile_width, s.tile_height, d_status=st)
    offsets = gs.gs_tile_offsets(keys, s.C, s.tile_width, s.tile_height, d_status=st)
    trace = torch.empty((keys.numel(), 8), dtype=torch.int32, device=DEV)
    rgb, alpha, last = gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"],
                                           d["opacities"], None, None, s.width, s.height, 16,
                                           offsets, ids, 1.0 / 255.0, 1e-4, d_status=st,
                                           trace=trace)
    b = gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"], None, None,
                            s.width, s.height, 16, offsets, ids, 1.0 / 255.0, alpha, last,
                            d["grad_render_colors"], d["grad_render_alphas"], trace=trace,
                            d_status=st)
    torch.cuda.synchronize()
    gs.check_status(st)
    assert I == keys.numel()
    CN, P = (s.C, s.N), (s.C, s.height, s.width)
    np.testing.assert_array_equal(out("tiles_per_gauss", np.int32, CN), tpg.cpu().numpy())
    np.testing.assert_array_equal(out("keys", np.int64, (I,)), keys.cpu().numpy())
    np.testing.assert_array_equal(out("flatten_ids", np.int32, (I,)), ids.cpu().numpy())
    np.testing.assert_array_equal(out("offsets", np.int32, offsets.shape),
                                  offsets.cpu().numpy())
    np.testing.assert_array_equal(out("render_colors", np.float32, P + (3,)), rgb.cpu().numpy())
    np.testing.assert_array_equal(out("render_alphas", np.float32, P + (1,)),
                                  alpha.cpu().numpy())
    np.testing.assert_array_equal(out("last_ids", np.int32, P), last.cpu().numpy())
    for name, shape in (("grad_means2d", CN + (2,)), ("grad_conics", CN + (3,)),
                        ("grad_colors", CN + (3,)), ("grad_opacities", CN)):
        x = b[name].cpu().numpy()
        np.testing.assert_allclose(out(name, np.float32, shape), x, rtol=1e-4,
                                   atol=1e-6 * (np.abs(x).max() + 1e-30), err_msg=name)
