"""Build libssd.so in-tree with nvcc for sm_103a (no cmake, parallel per translation unit).

Also builds libssd_xcheck.so, the test library: the same sources with the
cross-check kernels compiled in (SSD_CROSSCHECK: a CUDA-core rows kernel
and two other batch-1 GEMVs, selectable with SSD_OPT_GEMM_IMPL) for the
tests that compare kernels with each other.  Only the translation units
that use the flag are compiled twice."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libssd.so")
LIB_XCHECK = os.path.join(LIBDIR, "libssd_xcheck.so")
XCHECK_SOURCES = ("api.cu", "k_linear.cu")  # the translation units SSD_CROSSCHECK changes

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-ffp-contract=off", "--expt-relaxed-constexpr"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def build(force: bool = False, verbose: bool = False, extra: tuple = ()) -> str:
    os.makedirs(OBJDIR, exist_ok=True)
    nvcc = _nvcc()
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "ssd.h"))
    newest_header = max(os.path.getmtime(h) for h in headers)

    def compile_one(job):
        src, xcheck = job
        path = os.path.join(CSRC, src)
        obj = os.path.join(OBJDIR, src + (".xcheck.o" if xcheck else ".o"))
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(path), newest_header):
            return obj, ""
        if src.endswith(".cpp"):
            cmd = ["g++", *CXX_FLAGS, "-I", cuda_inc, "-c", path, "-o", obj]
        else:
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, *(["-DSSD_CROSSCHECK"] if xcheck else []), "-c", path, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    srcs = sources()
    jobs = [(src, False) for src in srcs] + [(src, True) for src in srcs if src in XCHECK_SOURCES]
    # the largest translation units first, so the parallel build ends sooner
    jobs.sort(key=lambda j: -os.path.getsize(os.path.join(CSRC, j[0])))
    with ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        results = dict(zip(jobs, ex.map(compile_one, jobs)))
    if verbose:
        for _, log in results.values():
            if log:
                print(log)
    prod = [results[(src, False)][0] for src in srcs]
    xcheck = [results[(src, src in XCHECK_SOURCES)][0] for src in srcs]

    def link(lib, objs):
        if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
            cmd = [nvcc, *ARCH, "-shared", "-o", lib, *objs]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")

    link(LIB, prod)
    link(LIB_XCHECK, xcheck)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True))
