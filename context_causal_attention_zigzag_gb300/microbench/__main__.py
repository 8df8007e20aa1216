"""Builds and runs the microbenchmarks on GPU 0: the tcgen05.mma rate with one
CTA per SM and cta_group::1 (mma_rate.cu), with CTA pairs and cta_group::2
(mma_rate_pair.cu), the bulk float32 reduction rate (reduce_rate.cu) and the
rate of bulk copies from L2 into shared memory (load_rate.cu).  ``--pair``,
``--single``, ``--reduce`` or ``--load`` runs only that one."""
import os
import subprocess
import sys
import tempfile

from .. import build as _build

HERE = os.path.dirname(os.path.abspath(__file__))


def run(src):
    exe = os.path.join(tempfile.gettempdir(), f"cpattn_{os.path.splitext(src)[0]}_{os.getpid()}")
    cmd = [_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
           "-I", _build.CSRC, "-o", exe, os.path.join(HERE, src)]
    subprocess.run(cmd, check=True)
    try:
        return subprocess.run([exe]).returncode
    finally:
        os.unlink(exe)


def main():
    srcs = ["mma_rate.cu", "mma_rate_pair.cu", "reduce_rate.cu", "load_rate.cu"]
    if "--pair" in sys.argv:
        srcs = ["mma_rate_pair.cu"]
    elif "--single" in sys.argv:
        srcs = ["mma_rate.cu"]
    elif "--reduce" in sys.argv:
        srcs = ["reduce_rate.cu"]
    elif "--load" in sys.argv:
        srcs = ["load_rate.cu"]
    rc = 0
    for s in srcs:
        rc |= run(s)
    sys.exit(rc)


if __name__ == "__main__":
    main()
