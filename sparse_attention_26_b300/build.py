"""Build libhattn.so (the CUDA library behind include/hattn.h) in-tree, for sm_103a.

    python -m sparse_attention_26_b300.build [--force] [--verbose]

Each .cu under csrc/ is compiled with nvcc -gencode arch=compute_103a,code=sm_103a
-O3 -lineinfo and linked into sparse_attention_26_b300/libhattn.so (shared
cudart, rpath to the CUDA toolkit).  Objects are cached under _build/.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libhattn.so")
SOURCES = ["abi.cu", "compress.cu", "indexer.cu", "topk.cu", "qprep.cu", "attention.cu",
           "merge.cu", "quant.cu", "hidden.cu"]
HEADERS = ["common.cuh", "kernels.h", os.path.join("..", "..", "include", "hattn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for c in [shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhattn")


def _cuda_lib_dir(nvcc):
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False):
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS]
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
                    "-fvisibility=hidden", "--expt-relaxed-constexpr", "-Xptxas", "-v" if verbose
                    else "-O3"]
    jobs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs + [__file__]):
            jobs.append([nvcc] + flags + ["-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4) or 1) as ex:
        for out in ex.map(run, jobs):
            if verbose and out:
                print(out)
    if force or jobs or _stale(LIB, objs):
        run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", LIB] + objs +
            ["-Xlinker", "-rpath=" + _cuda_lib_dir(nvcc)])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
