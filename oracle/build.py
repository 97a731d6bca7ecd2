"""Compile the CPU oracle (test infrastructure) into oracle/libspecoracle.so."""

from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def oracle_lib_path() -> str:
    return os.path.join(_HERE, "libspecoracle.so")


def build_oracle(src: str | None = None, out: str | None = None) -> str:
    """gcc -O2, no fast-math, OpenMP over rows. Returns the library path."""
    src = src or os.path.join(_HERE, "spec_oracle.c")
    out = out or oracle_lib_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle())
