"""Build the GDN CUDA library (libgdn.so, sm_103a) in-tree with nvcc."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libgdn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def sources():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))] + [
        os.path.join(HERE, "..", "include", "gdn.h")]


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile csrc/gdn_lib.cu into libgdn.so next to this file (skips if up to date)."""
    newest = max(os.path.getmtime(p) for p in sources())
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest and not extra:
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["nvcc", *ARCH, *FLAGS, *extra, "-o", tmp, os.path.join(CSRC, "gdn_lib.cu")]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
