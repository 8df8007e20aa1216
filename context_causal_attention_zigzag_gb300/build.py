"""Builds libcpattn.so in-tree for sm_103a with nvcc.

Each translation unit under csrc/ compiles in parallel to _build/*.o, then
one shared library is linked next to this file.  CUDA runtime is linked
statically, so the library only needs the driver at load time.
"""
import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = _BUILD = os.path.join(PKG, "_build")
LIB = _LIB = os.path.join(PKG, "libcpattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def mutant_lib_path(mutation: int) -> str:
    """Where the build with planted mistake ``mutation`` puts its library."""
    return os.path.join(PKG, f"_build_mut{int(mutation)}", "libcpattn.so")


def build(force: bool = False, verbose: bool = False, extra_flags=(), mutation: int = 0) -> str:
    """Compiles every translation unit under csrc/ and links libcpattn.so.
    ``mutation`` > 0 compiles planted mistake number ``mutation`` (see
    CPATTN_MUTATION in csrc/cpattn_internal.h) into a library of its own
    folder, for the mutation tests; the regular build is 0."""
    BUILD = _BUILD if mutation == 0 else os.path.dirname(mutant_lib_path(mutation))
    LIB = _LIB if mutation == 0 else mutant_lib_path(mutation)
    if mutation:
        extra_flags = tuple(extra_flags) + (f"-DCPATTN_MUTATION={int(mutation)}",)
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    objs = []
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
        if verbose and (p.stdout or p.stderr):
            print(p.stdout + p.stderr, flush=True)

    if jobs:
        with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lrt", "-ldl", "-lpthread"]
        run(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
