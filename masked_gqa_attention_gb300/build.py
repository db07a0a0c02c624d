"""Build the CUDA libraries for sm_103a with nvcc, in-tree.

Each translation unit under csrc/ compiles in parallel to an object file;
the objects link into two libraries under masked_gqa_attention_gb300/_lib:
  * libmgqa.so        -- the product library;
  * libmgqa_debug.so  -- the same sources with MGQA_DEBUG: device-side bounds
                         checks, event counters and an injectable pipeline
                         stall (include/masked_gqa_attn_debug.h); test equipment.
The CUDA runtime is linked statically; the driver entry point used for TMA
tensor maps is fetched at run time, so the libraries load on machines
without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libmgqa.so")
LIB_DEBUG = os.path.join(OUT_DIR, "libmgqa_debug.so")
OBJ_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]
# variant -> (library, object directory, extra flags)
VARIANTS = {
    "release": (LIB, OBJ_DIR, []),
    "debug": (LIB_DEBUG, os.path.join(OBJ_DIR, "debug"), ["-DMGQA_DEBUG=1"]),
}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(os.path.dirname(PKG), "include", "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(),
          variants=("release", "debug")) -> str:
    """Compile and link the requested variants (both by default); returns the
    product library's path."""
    todo = [v for v in variants if force or not up_to_date(VARIANTS[v][0])]
    if not todo:
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    srcs = _sources()

    def compile_one(job):
        variant, src = job
        _, obj_dir, flags = VARIANTS[variant]
        obj = os.path.join(obj_dir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *flags, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)} ({variant}):\n"
                               f"{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(f"[{variant}] {os.path.basename(src)}\n{r.stdout}{r.stderr}")
        return obj

    for v in todo:
        os.makedirs(VARIANTS[v][1], exist_ok=True)
    jobs = [(v, src) for v in todo for src in srcs]
    workers = max(1, min(len(jobs), os.cpu_count() or 8))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(compile_one, jobs))
    for v in todo:
        lib = VARIANTS[v][0]
        vobjs = [o for (vv, _), o in zip(jobs, objs) if vv == v]
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *vobjs, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({v}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    variants = ("release",) if "--release-only" in sys.argv else ("release", "debug")
    print(build(force="--force" in sys.argv, verbose=True, variants=variants,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
