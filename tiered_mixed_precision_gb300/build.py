"""Build libfade.so in-tree for sm_103a with nvcc (no cmake, no torch extension machinery).

Each translation unit is compiled in parallel; the objects are linked into
``tiered_mixed_precision_gb300/_build/libfade.so``. Host code is compiled without
floating-point contraction so that the host-side RoPE frequency math rounds as written.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")   # FADE_DEBUG=1: device checks on hot paths
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(BUILD, "libfade.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-ffp-contract=off",
           "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfade")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def build(verbose: bool = False, force: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile every .cu under csrc/ and link libfade.so; returns the library path. debug:
    the FADE_DEBUG=1 variant (index checks on every compacted row and attention tile that
    record a code in the layer's status word) in its own directory."""
    out_dir = BUILD_DEBUG if debug else BUILD
    lib_path = os.path.join(out_dir, "libfade.so")
    if debug:
        extra_flags = (*extra_flags, "-DFADE_DEBUG=1")
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    hdrs = _headers()
    objs, jobs = [], []
    for src in sources():
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src, *hdrs, __file__]):
            cmd = [nvcc, *ARCH, *NVFLAGS, *extra_flags, "-c", src, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(lib_path, objs):
        run([nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", lib_path])
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
