"""Build libqlin.so (the CUDA kernels and the C ABI) for sm_103a, in-tree.

    python -m activation_quantization_quantize_b300.build [--force]

nvcc cross-compiles without a GPU; the library links the CUDA runtime
statically and resolves driver entry points at run time, so it loads on a
machine without a GPU (every call then fails with QLIN_ERR_CUDA).
"""
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libqlin.so")
ROOT = os.path.dirname(HERE)

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "qlin.h")])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libqlin.so if any source is newer than it; return its path."""
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in sources())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [NVCC, *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"),
           os.path.join(CSRC, "qlin_lib.cu"), "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
