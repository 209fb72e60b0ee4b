"""In-tree build of the CUDA libraries (sm_103a only).

libspc.so      <- bit_kv_cache_spc_gb300/csrc/*.cu  (the product: the C-ABI of include/spc.h)
libspc_synth.so <- synth/synth.cu                   (the seeded input generator's GPU twin)

Each translation unit is compiled in parallel, then linked with nvcc -shared.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(PKG, "_build")
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]

LIBSPC = os.path.join(PKG, "libspc.so")
LIBSYNTH = os.path.join(ROOT, "synth", "libspc_synth.so")


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _compile_link(sources, headers, target, verbose=False, extra=()):
    if not _stale(target, list(sources) + list(headers)):
        return target
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    objs = []
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or p.returncode != 0):
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = target + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs])  # static cudart: no runtime path needed
    os.replace(tmp, target)
    return target


def build(verbose: bool = False):
    csrc = os.path.join(PKG, "csrc")
    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")))
    hdrs = sorted(glob.glob(os.path.join(csrc, "*.cuh"))) + [os.path.join(ROOT, "include", "spc.h")]
    _compile_link(srcs, hdrs, LIBSPC, verbose)
    synth_src = os.path.join(ROOT, "synth", "synth.cu")
    if os.path.exists(synth_src):
        _compile_link([synth_src], [], LIBSYNTH, verbose)
    return LIBSPC


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
