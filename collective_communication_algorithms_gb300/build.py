"""Build libhc.so (and libhc.a) in-tree with nvcc for sm_103a.

Output: collective_communication_algorithms_gb300/_lib/libhc.so
Sources are compiled in parallel, one translation unit per process, then
linked; the CUDA runtime is linked statically so the library carries no
dependency on a particular libcudart.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT, "libhc.so")
ARCHIVE = os.path.join(OUT, "libhc.a")
SOURCES = ["hc_kernels.cu", "hc_fused_ring.cu", "hc_fused_rhd.cu", "hc_fused_pipe.cu",
           "hc_fused_hier.cu", "hc_sched.cpp", "hc_api.cpp", "hc_graph.cpp", "hc_static_scratch.cu",
           "hc_trace.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhc")


def _flags(src):
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
    if src.endswith(".cu"):
        return common + ARCH + ["-lineinfo", "-Xptxas", "-warn-spills"]
    return common + ["-x", "c++"]


def _compile(src, obj):
    cmd = [nvcc(), *_flags(src), "-c", os.path.join(CSRC, src), "-o", obj]
    subprocess.run(cmd, check=True)
    return obj


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    deps = [os.path.join(CSRC, s) for s in SOURCES]
    deps += [os.path.join(CSRC, "hc_internal.h"), os.path.join(CSRC, "hc_device.cuh"),
             os.path.join(ROOT, "include", "hc.h")]
    if not force and not _stale(LIB, deps):
        return LIB
    objs = [os.path.join(OUT, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(_compile, SOURCES, objs))
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.run([nvcc(), "-shared", *ARCH, "-cudart", "static", *objs, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    if os.path.exists(ARCHIVE):
        os.remove(ARCHIVE)
    subprocess.run(["ar", "rcs", ARCHIVE, *objs], check=True)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
