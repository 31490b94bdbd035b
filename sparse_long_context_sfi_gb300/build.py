"""Build the in-tree shared libraries with nvcc for sm_103a.

  sparse_long_context_sfi_gb300/libsfi.so   the C-ABI library (include/sfi.h)
  synth/libsynth.so                          the GPU twin of the seeded input generator

Translation units compile in parallel into _build/ next to this file; the CUDA runtime is
linked statically and the driver's tensor-map encoder is resolved at run time, so the
libraries need no libcuda at link time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libsfi.so")
SYNTH_SRC = os.path.join(ROOT, "synth", "csrc", "synth_gen.cu")
SYNTH_LIB = os.path.join(ROOT, "synth", "libsynth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
SOURCES = ["attn.cu", "select.cu", "refine.cu", "kvops.cu", "api.cpp"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_sfi(force: bool = False, verbose: bool = False, extra=()) -> str:
    out_dir = os.path.join(PKG, "_build")
    os.makedirs(out_dir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "sfi.h"))
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src + ".o")
        if force or _stale(o, [s, *headers]):
            cmd = [nvcc(), *ARCH, *COMMON, *extra, "-c", s, "-o", o]
            if src.endswith(".cu") and verbose:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for log in ex.map(_run, jobs):
            if verbose and log.strip():
                print(log)
    objs = [os.path.join(out_dir, s + ".o") for s in SOURCES]
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        _run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


def build_synth(force: bool = False) -> str:
    if force or _stale(SYNTH_LIB, [SYNTH_SRC]):
        tmp = SYNTH_LIB + f".tmp{os.getpid()}"
        _run([nvcc(), *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", SYNTH_SRC,
              "-o", tmp])
        os.replace(tmp, SYNTH_LIB)
    return SYNTH_LIB


def build_all(force: bool = False, verbose: bool = False):
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        a = ex.submit(build_sfi, force, verbose)
        b = ex.submit(build_synth, force)
        return a.result(), b.result()


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv, verbose="-v" in sys.argv))
