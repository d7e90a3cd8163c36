"""Build libq4_0.so in-tree with nvcc for sm_103a.

The four translation units compile in parallel; the shared library links the
CUDA runtime statically, so it loads on a machine without a GPU (the driver
is reached at run time through cudaGetDriverEntryPointByVersion).  ptxas
register/spill reports go to ``_build/ptxas.log``.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "lib", "libq4_0.so")
SOURCES = ["api.cu", "quantize.cu", "gemv.cu", "gemv_tc.cu", "gemm.cu", "noalloc.cu", "pad.cu"]
HEADERS = ["q4_0_internal.h", "q4_0_ptx.cuh"]
PUBLIC_HEADER = os.path.join(os.path.dirname(HERE), "include", "q4_0.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libq4_0.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src), PUBLIC_HEADER] + [os.path.join(CSRC, h) for h in HEADERS]
    if _stale(obj, deps):
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(os.path.join(BUILD, os.path.splitext(src)[0] + ".ptxas.log"), "w") as f:
            f.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
    return obj


def build(force: bool = False) -> str:
    """Compile (if stale) and return the path of libq4_0.so."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    if _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as out:
        for src in SOURCES:
            p = os.path.join(BUILD, os.path.splitext(src)[0] + ".ptxas.log")
            if os.path.exists(p):
                out.write(open(p).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
