"""Builds libbsq.so in-tree: one nvcc job per translation unit, in parallel,
for sm_103a only, then one shared-object link (static cudart, no -lcuda: the
tensor-map encoder is resolved through the runtime at first use)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbsq.so")
SOURCES = ["bsq_api.cu", "quantize.cu", "gemv.cu", "gemm.cu", "dequant.cu"]
HEADERS = ["bsq_device.cuh", "bsq_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "bsq.h")]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append([cc, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed: " + " ".join(cmd))
        os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, defines, rebuilt=("bsq_api.cu", "quantize.cu")) -> str:
    """A separately named copy of the library (lib<name>.so in _build_<name>/)
    whose `rebuilt` translation units are compiled with extra preprocessor
    defines; the others are the regular build's objects.  Used by tests for
    compile-time test hooks (a short wait limit, a skipped barrier arrival),
    never by the product path."""
    build()
    out_dir = os.path.join(PKG, f"_build_{name}")
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = [f"-D{d}" for d in defines]
    objs, jobs = [], []
    for src in SOURCES:
        if src in rebuilt:
            o = os.path.join(out_dir, src.replace(".cu", ".o"))
            jobs.append([cc, *NVCC_FLAGS, *flags, "-c", os.path.join(CSRC, src), "-o", o])
        else:
            o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for r in ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs):
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError("nvcc failed for variant " + name)
    lib = os.path.join(out_dir, f"lib{name}.so")
    r = subprocess.run([cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", lib, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed for variant " + name)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
    print(LIB)
