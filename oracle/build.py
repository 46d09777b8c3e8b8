"""Compile the CPU oracle (``fd_oracle.c``) into ``oracle/_build/libfd_oracle.so``.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The flags matter: the
key encoder runs in IEEE binary32 and must not be contracted into fused
multiply-adds (gcc contracts by default on aarch64), nor use fast-math.
Run ``python -m oracle.build`` or let the package build on first use.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fd_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard", "-Wall", "-Wextra"]


def library_path() -> str:
    return os.path.join(OUT_DIR, "libfd_oracle.so")


def is_stale() -> bool:
    out = library_path()
    return (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(SRC)


def build(verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    out = library_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
