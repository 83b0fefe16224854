"""Build libmoe.so in-tree with nvcc for sm_103a (no JIT cache, no torch extension)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmoe.so")
SOURCES = ["api.cu", "decode.cu", "scalar.cu", "noalloc.cu", "batched.cu", "grouped.cu", "gemv.cu", "hybrid.cu", "qpack.cpp"]
HEADERS = ["layout.h", "policy.h", "host.h", "grouped.h", "qpack.h", "attr.h"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_cmd(out: str = LIB, extra=()) -> list[str]:
    return (["nvcc", ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
             "-Xcompiler", "-Wall", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
             "-o", out] + list(extra) + [os.path.join(CSRC, s) for s in SOURCES])


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [
        os.path.join(ROOT, "include", h) for h in ("moe.h", "hybrid.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile when forced or stale. The library is written to a per-process temporary file and
    renamed into place, so ranks that build at the same time never load a half-written file."""
    if force or stale():
        extra = ["-Xptxas", "-v"] if verbose else []
        tmp = f"{LIB}.tmp{os.getpid()}"
        try:
            subprocess.run(nvcc_cmd(tmp, extra), check=True)
            os.replace(tmp, LIB)
        finally:
            if os.path.exists(tmp):
                os.remove(tmp)
    return LIB


if __name__ == "__main__":
    import sys
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
