"""Builds libgs_splat_gb300.so in-tree from csrc/*.cu for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked with the
static CUDA runtime into one shared library beside this file.  No fast-math
flags: the tile bounds need IEEE division and exact floor/ceil, and the
raster kernels choose their fast intrinsics explicitly.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgs_splat_gb300.so")
# the range-checking build (GS_DEBUG_BOUNDS): the same sources, reporting
# GS_ERR_OUT_OF_BOUNDS where an index read from the inputs is out of range
LIB_DEBUG = os.path.join(HERE, "libgs_splat_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(HERE, "..", "include", "gs_splat.h")]


def _variants(debug):
    out = [(LIB, os.path.join(BUILD, "release"), [])]
    if debug:
        out.append((LIB_DEBUG, os.path.join(BUILD, "debug"), ["-DGS_DEBUG_BOUNDS"]))
    return out


def build(force: bool = False, verbose: bool = False, extra=(), debug: bool = True) -> str:
    """Compiles every translation unit of the library (and, with debug, of
    its range-checking build) in parallel and links each.  Returns the path
    of the release library."""
    srcs = sources()
    newest = max(os.path.getmtime(p) for p in _deps())
    todo = [(lib, d, f) for lib, d, f in _variants(debug)
            if force or extra or not os.path.exists(lib) or os.path.getmtime(lib) < newest]
    if not todo:
        return LIB
    nvcc = _nvcc()

    def compile_one(job):
        src, objdir, flags = job
        os.makedirs(objdir, exist_ok=True)
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    jobs = [(src, d, f) for _, d, f in todo for src in srcs]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for k, (lib, _, _) in enumerate(todo):
        part = objs[k * len(srcs):(k + 1) * len(srcs)]
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", *part, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith(("-X", "--", "-D"))]
    print(build(force="--force" in sys.argv, verbose=True,
                extra=[a for a in extra if a != "--force"]))
