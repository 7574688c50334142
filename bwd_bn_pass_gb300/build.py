"""Build libgbnorm.so in-tree with nvcc for sm_103a (GB300).

Each .cu file is compiled to an object in parallel, then linked into a
shared library next to this file.  No CMake, no torch extension: the library
exports a plain C ABI and is loaded with ctypes, so it does not depend on the
installed PyTorch version.

    python -m bwd_bn_pass_gb300.build          # or build_library()
"""

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libgbnorm.so"

SOURCES = ["abi.cu", "bn_kernels.cu", "rms_kernels.cu", "ln_kernels.cu",
           "row_common.cu", "noalloc.cu", "bn_fused.cu", "bn_small.cu", "fwd_kernels.cu",
           "bn_nhwc.cu", "selftest.cu"]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE,
                "-I", CSRC]


def nvcc_path():
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"),
                 "/usr/local/cuda"):
        if cand:
            p = os.path.join(cand, "bin", "nvcc")
            if os.path.exists(p):
                return p
    p = shutil.which("nvcc")
    if p is None:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return p


def library_path():
    return os.path.join(HERE, LIB_NAME)


def build_library(verbose=False, extra_flags=()):
    """Compile and link; returns the library path.  Raises on failure."""
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH_FLAGS, *COMMON_FLAGS, *extra_flags, "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text.strip():
            print(text, flush=True)
    if failed:
        msg = "\n".join(f"--- {s} ---\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = library_path() + ".tmp"
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, library_path())
    return library_path()


if __name__ == "__main__":
    build_library(verbose="-v" in sys.argv)
    print(library_path())
