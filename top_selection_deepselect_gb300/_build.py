"""Build libds_topk.so in-tree with nvcc for sm_103a (no CMake, one translation unit)."""
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libds_topk.so")
SOURCES = [os.path.join(CSRC, "ds_topk.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ds_device.cuh"), os.path.join(INCLUDE, "ds_topk.h")]

# No fast-math and no flush-to-zero: the prefilter compares denormals exactly.
NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC", "-shared", "--expt-relaxed-constexpr"]


def nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def needs_build(out=LIB_PATH):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force=False, verbose=False, extra_flags=()):
    """Compile the CUDA library if it is missing or older than its sources."""
    if not force and not needs_build():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + NVCC_FLAGS + list(extra_flags) + ["-I", INCLUDE, "-o", tmp] + SOURCES
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
