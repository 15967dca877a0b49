"""Build libspecverify.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu translation unit compiles in parallel, then nvcc links them into one
shared library next to this file.  No cmake, no torch extension machinery.

build(variant="bounds") makes libspecverify_bounds.so instead: the same
sources with -DSV_BOUNDS, whose kernels check every computed index before
the access and record the bad ones (read back with spec_debug_bounds); the
GPU tests run their guard-region cases through it as well.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libspecverify.so")
VARIANTS = {None: (BUILD, LIB, []),
            "bounds": (os.path.join(HERE, "_build_bounds"),
                       os.path.join(HERE, "libspecverify_bounds.so"), ["-DSV_BOUNDS"])}
SOURCES = ["api.cu", "chain_stochastic.cu", "greedy.cu", "rollback.cu", "kv_policy.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "specverify.h"))
    files.append(os.path.abspath(__file__))
    return files


def build(force=False, verbose_ptxas=False, variant=None):
    """Compile and link; skip when the library is newer than every source."""
    build_dir, lib, extra = VARIANTS[variant]
    if not force and os.path.exists(lib):
        newest = max(os.path.getmtime(f) for f in _deps())
        if os.path.getmtime(lib) >= newest:
            return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
             "-I", INCLUDE, "-I", CSRC, *extra]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    # extra nvcc flags for measurement and tuning builds
    flags += os.environ.get("SPECVERIFY_NVCC_FLAGS", "").split()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas:
        for _, err in results:
            sys.stderr.write(err)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp"
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                variant="bounds" if "--bounds" in sys.argv else None))
