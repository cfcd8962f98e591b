"""Build libgq.so (the C-ABI library of include/gq.h) in-tree with nvcc for sm_103a.

Flags: one -gencode (compute_103a -> sm_103a), -O3, -lineinfo, --fmad=false (no
multiply-add contraction anywhere, on top of the explicit _rn intrinsics), no fast-math.
The runtime is linked as a shared library so the process shares one libcudart with
PyTorch.  Translation units compile in parallel.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libgq.so")
BUILD = os.path.join(HERE, "_build")
SOURCES = ["gq_pipe_f16.cu", "gq_pipe_f32.cu", "gq_queue_f16.cu", "gq_queue_f32.cu", "gq_fused_f16.cu", "gq_fused_f32.cu",
           "gq_kernels.cu", "gq_api.cu"]
HEADERS = ["gq_device.cuh", "gq_internal.h", "gq_fused.cuh", "gq_queue.cuh", "gq_pipe.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-Wall", "-I" + os.path.join(ROOT, "include")]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return path


def cuda_lib_dir():
    base = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    for d in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
              os.path.join("targets", "x86_64-linux", "lib")):
        if os.path.exists(os.path.join(base, d, "libcudart.so")):
            return os.path.join(base, d)
    return os.path.join(base, "lib64")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose_ptxas=False, extra_flags=(), out=None):
    """Compile and link libgq.so (to `out`, default in the package directory).  extra_flags
    go to every nvcc compile (e.g. -D settings of the kernels' launch bounds)."""
    lib = out or LIB
    build_dir = os.path.join(os.path.dirname(lib), "_build") if out else BUILD
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [
        os.path.join(ROOT, "include", h) for h in ("gq.h", "gq_testing.h")]
    if not force and not _stale(lib, deps):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + list(extra_flags)

    def compile_one(src):
        obj = os.path.join(build_dir, src + ".o")
        cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    tmp = lib + ".tmp%d" % os.getpid()
    libdir = cuda_lib_dir()
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-L" + libdir, "-Xlinker", "-rpath=" + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    if verbose_ptxas:
        return lib, "\n".join(err for _, err in results)
    return lib


if __name__ == "__main__":
    out = build(force=True, verbose_ptxas=True)
    print(out[0])
    print(out[1])
