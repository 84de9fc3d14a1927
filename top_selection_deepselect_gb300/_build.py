"""Build libds_topk.so in-tree with nvcc for sm_103a (no CMake, one translation unit)."""
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libds_topk.so")
SOURCES = [os.path.join(CSRC, f) for f in ("ds_topk.cu", "ds_kernels_fp32.cu", "ds_kernels_bf16.cu",
                                         "ds_kernels_fp16.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ds_device.cuh"), os.path.join(CSRC, "ds_kernel.cuh"),
                  os.path.join(CSRC, "ds_stream.cuh"),
                  os.path.join(INCLUDE, "ds_topk.h")]

# No fast-math and no flush-to-zero: the prefilter compares denormals exactly.
NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


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
    """Compile the CUDA library if it is missing or older than its sources.

    The translation units compile in parallel into _build/, then nvcc links
    them into the shared library."""
    if not force and not needs_build():
        return LIB_PATH
    objdir = os.path.join(PKG, "_build")
    os.makedirs(objdir, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(objdir, os.path.splitext(os.path.basename(src))[0] + ".o")
        objs.append(obj)
        cmd = [nvcc()] + NVCC_FLAGS + list(extra_flags) + ["-I", INCLUDE, "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd)))
    failed = [src for src, p in procs if p.wait() != 0]
    if failed:
        raise RuntimeError("nvcc failed on " + ", ".join(failed))
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.run([nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp]
                   + objs, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
