"""Build libmsda.so (the CUDA kernels and the C ABI) in-tree, for sm_103a, and
beside it libmsda_debug.so (the same with every kernel access checked) and
libmsda_probes.so (line-rate measurement kernels, used by bench.py).

    python scale_deformable_attention_06_b300/build.py [--force] [--verbose]

The library links the shared CUDA runtime (libcudart.so.13), so it shares the
runtime state (current device, streams) of the process that loads it.
"""
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmsda.so")
PROBES_LIB = os.path.join(PKG, "libmsda_probes.so")
DEBUG_LIB = os.path.join(PKG, "libmsda_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(out, srcs, verbose=False, extra=()):
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
           "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64", "-I", INCLUDE,
           "--expt-relaxed-constexpr", *extra, "-o", out + ".tmp", *srcs]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)


def build_probes(force=False):
    """libmsda_probes.so: the line-rate measurement kernels (include/msda_probes.h)."""
    srcs = sorted(glob.glob(os.path.join(CSRC, "probes", "*.cu")))
    deps = srcs + [os.path.join(INCLUDE, "msda_probes.h"), os.path.abspath(__file__)]
    if force or not os.path.exists(PROBES_LIB) or any(os.path.getmtime(p) > os.path.getmtime(PROBES_LIB)
                                                      for p in deps):
        _compile(PROBES_LIB, srcs, extra=("-Xcompiler", "-fvisibility=default"))
    return PROBES_LIB


def build_debug(force=False):
    """libmsda_debug.so: the same sources with -DMSDA_DEBUG (every kernel access
    checked against its tensor's extent, bad ones counted and skipped;
    include/msda_debug.h)."""
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    if force or not os.path.exists(DEBUG_LIB) or any(os.path.getmtime(p) > os.path.getmtime(DEBUG_LIB) for p in deps):
        _compile(DEBUG_LIB, sources(), extra=("-DMSDA_DEBUG",))
    return DEBUG_LIB


def build(force=False, verbose=False, extra=()):
    build_probes(force)
    build_debug(force)
    if not force and not _stale():
        return LIB
    _compile(LIB, sources(), verbose, extra)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
