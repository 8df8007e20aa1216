"""Builds and runs the tcgen05.mma rate microbenchmark (mma_rate.cu) on GPU 0."""
import os
import subprocess
import sys
import tempfile

from .. import build as _build

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    exe = os.path.join(tempfile.gettempdir(), f"cpattn_mma_rate_{os.getpid()}")
    cmd = [_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
           "-I", _build.CSRC, "-o", exe, os.path.join(HERE, "mma_rate.cu")]
    subprocess.run(cmd, check=True)
    try:
        rc = subprocess.run([exe]).returncode
    finally:
        os.unlink(exe)
    sys.exit(rc)


if __name__ == "__main__":
    main()
