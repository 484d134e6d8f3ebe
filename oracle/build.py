"""Builds the oracle's shared library (plain C, fp64, OpenMP) in-tree.

Test infrastructure: compiled by ``__graft_entry__.build()`` so the checker
exists on every machine, used only by tests, smoke and the CPU baseline."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mc_oracle.c")


def library_path() -> str:
    return os.path.join(_HERE, "libmc_oracle.so")


def build(force: bool = False) -> str:
    out = library_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add contraction, so both x86 and
    # Arm hosts evaluate every expression with the same roundings.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
