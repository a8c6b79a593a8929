"""Build libpkv.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel, then linked into
paged_kv_cache_137_gb300/_lib/libpkv.so (static CUDA runtime).  A build is
skipped when the library is newer than every source and header and was built
for this machine's architecture.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libpkv.so")
STAMP = os.path.join(OUT_DIR, "build_arch.txt")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-Xptxas", "-warn-spills"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-Wall"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    if open(STAMP).read().strip() != platform.machine():
        return False
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) \
        + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return all(os.path.getmtime(d) <= t for d in deps)


def _compile(src: str, obj: str) -> tuple[str, str]:
    if src.endswith(".cu"):
        cmd = [nvcc(), *ARCH, *CUDA_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    else:
        cxx = shutil.which("g++") or "g++"
        cuda_inc = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "include")
        cmd = [cxx, *CXX_FLAGS, "-I", INCLUDE, "-I", CSRC, "-I", cuda_inc, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return src, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libpkv.so if needed; return its path."""
    if not force and _up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    objs_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(objs_dir, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(objs_dir, os.path.basename(s) + ".o") for s in srcs]
    workers = max(1, min(len(srcs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        for src, log in ex.map(lambda p: _compile(*p), zip(srcs, objs)):
            if verbose and log.strip():
                print(f"[{os.path.basename(src)}]\n{log}")
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(platform.machine())
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
