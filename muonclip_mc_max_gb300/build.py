"""In-tree build of the CUDA library ``libmc_max.so`` for sm_103a.

Each translation unit under ``csrc/`` is compiled by nvcc in parallel with
``-gencode arch=compute_103a,code=sm_103a`` and linked into one shared
library next to this file (git-ignored).  No CMake, no torch extension
machinery: the library exposes the plain C ABI of ``include/mc_max.h``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_BUILD = os.path.join(_ROOT, "_build", "mc_max")
SOURCES = ["abi.cu", "gemm.cu", "scan.cu", "elementwise.cu", "attn.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def library_path() -> str:
    return os.path.join(_HERE, "libmc_max.so")


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _deps_mtime() -> float:
    paths = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC)]
    paths.append(os.path.join(_ROOT, "include", "mc_max.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    out = library_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= _deps_mtime():
        return out
    os.makedirs(_BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", os.path.join(_ROOT, "include")]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(_BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc] + common + ["-c", os.path.join(_CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))
