"""Build the GPU library ``libvqx.so`` in-tree with nvcc for sm_103a.

The library is a plain C-ABI shared object (no PyTorch in it): the CUDA
runtime is linked statically and its symbols are kept private, so the only
exported names are the ``vqx_*`` entry points of ``include/vqx.h``.

Device code is compiled with ``--fmad=false`` and host code with
``-ffp-contract=off``: no multiply may be fused with an add anywhere on the
path, because the per-pixel terms must be the CPU's separately rounded
products and the host conclusion the CPU's separately rounded divisions.
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD_DIR, "libvqx.so")
SOURCES = [os.path.join(CSRC, "vqx_plane_stats.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "vqx_kernels.cuh"), os.path.join(CSRC, "vqx_ordered.cuh"),
                     os.path.join(CSRC, "vqx_hvs.cuh"),
                     os.path.join(INCLUDE, "vqx.h"),
                     os.path.abspath(__file__)]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def command(out, verbose_ptxas=False):
    cmd = [
        nvcc(),
        ARCH,
        "-O3",
        "-std=c++17",
        "-lineinfo",
        "--fmad=false",
        "-Xcompiler=-fPIC,-ffp-contract=off,-fno-fast-math",
        "-Xlinker=--exclude-libs,ALL",
        "-shared",
        "-cudart=static",
        "-I" + INCLUDE,
        "-I" + CSRC,
        "-o",
        out,
        *SOURCES,
    ]
    if verbose_ptxas:
        cmd.insert(2, "-Xptxas=-v")
    return cmd


def up_to_date(out=LIB):
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(p) <= t for p in DEPENDS)


def build_library(force=False, verbose_ptxas=False):
    """Compile ``libvqx.so`` unless it is newer than every source."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.run(command(tmp, verbose_ptxas), check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
