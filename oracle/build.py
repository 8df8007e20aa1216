"""Builds the CPU oracle (plain C, fp64, OpenMP) into oracle/_build/.

Test infrastructure: the product library never links this.  ``mutation`` > 0
compiles one of the planted mistakes used by the mutation tests into a
separate library file; the regular build always uses 0.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cpattn_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")


def lib_path(mutation: int = 0) -> str:
    name = "liboracle.so" if mutation == 0 else f"liboracle_mut{mutation}.so"
    return os.path.join(OUT_DIR, name)


def build(mutation: int = 0, force: bool = False) -> str:
    out = lib_path(mutation)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           f"-DORACLE_MUTATION={int(mutation)}", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
