"""Builds libvcd.so in-tree: the CUDA kernels and the C ABI, for sm_103a only.

    python -m varlen_causal_depthwise_gb300.build

Each translation unit compiles in parallel with nvcc; the objects link into a
shared library with the CUDA runtime linked statically, so the library needs no
CUDA runtime of its own at load time and cooperates with torch's device memory
and streams through the driver.
"""
import concurrent.futures
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libvcd.so")
BUILD = os.path.join(PKG, "_build")
SOURCES = ["vcd_fwd.cu", "vcd_bwd.cu", "vcd_capi.cu", "vcd_noalloc.cu", "vcd_stream.cu"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}"]


def _compile(src, defines=(), verbose=False):
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    return obj


def build(out=OUT, defines=(), verbose=False):
    """Compile every kernel and the C ABI into ``out``; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, defines, verbose), SOURCES))
    subprocess.run([NVCC, *ARCH, "-shared", "-o", out, *objs], check=True)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
