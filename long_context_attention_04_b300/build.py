"""Build liblca.so (the CUDA library behind include/lca.h) for sm_103a with nvcc."""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "liblca.so")
MAIN_SRC = os.path.join(PKG, "csrc", "lca.cu")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-Xptxas", "-v",
]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(PKG, "csrc", "*.cu*"))) + [os.path.join(ROOT, "include", "lca.h")]


def stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if a source is newer than it (or when forced); returns its path."""
    if not force and not stale():
        return LIB_PATH
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [nvcc, *NVCC_FLAGS, "-o", tmp, MAIN_SRC]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(PKG, "build.log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + proc.stdout + proc.stderr)
    if proc.returncode != 0:
        raise RuntimeError("nvcc failed building liblca.so:\n" + proc.stderr[-6000:])
    if verbose:
        print(proc.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
