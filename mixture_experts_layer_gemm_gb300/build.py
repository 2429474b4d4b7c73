"""Build ``libmoe_layer.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` compiles to an object in ``_build/`` (in parallel), then the
objects link into ``libmoe_layer.so`` next to this file.  The CUDA runtime is
linked statically, so the library needs nothing from torch at load time.

``build(trace=True)`` makes the tile-trace build instead: the same sources with
``MOE_TILE_TRACE`` defined (per-tile timestamps in the tensor-core kernels),
objects in ``_build_trace/``, linked into ``libmoe_layer_trace.so``.  Only the
tile-trace tool loads it.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_layer.so")
BUILD_TRACE = os.path.join(HERE, "_build_trace")
LIB_TRACE = os.path.join(HERE, "libmoe_layer_trace.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def nvcc():
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "moe_layer.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src, extra, verbose, build_dir=BUILD):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    if (os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
            and os.path.getmtime(obj) >= _headers_mtime()):
        return obj, ""
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    return obj, (r.stderr if verbose else "")


def build(force: bool = False, verbose: bool = False, extra=(), trace: bool = False) -> str:
    build_dir, lib = (BUILD_TRACE, LIB_TRACE) if trace else (BUILD, LIB)
    extra = list(extra) + (["-DMOE_TILE_TRACE"] if trace else [])
    os.makedirs(build_dir, exist_ok=True)
    if force:
        for f in os.listdir(build_dir):
            os.remove(os.path.join(build_dir, f))
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, verbose, build_dir), srcs))
    objs = [o for o, _ in results]
    for _, log in results:
        if log:
            sys.stderr.write(log)
    if (force or not os.path.exists(lib)
            or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs)):
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force="--force" in sys.argv, verbose=verbose or bool(extra), extra=extra))
