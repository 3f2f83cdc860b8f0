"""Build the in-tree CUDA libraries for sm_103a with nvcc.

* bit_expert_ffn_warp_b300/libbitmoe.so -- the kernels behind include/bitmoe.h
* synth/libsynth.so                     -- the device twin of the input generator

Objects go to ``_build/``; a library is rebuilt when any of its sources or
headers is newer than it.  ``python bit_expert_ffn_warp_b300/build.py [-f] [-v] [--ptxas]``
(run it by path: importing the package itself needs the built library).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]

LIBBITMOE = os.path.join(PKG, "libbitmoe.so")
LIBSYNTH = os.path.join(ROOT, "synth", "libsynth.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hdrs + [os.path.join(ROOT, "include", "bitmoe.h")]


def _stale(target, inputs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)


def _compile(src, obj, verbose, ptxas_v):
    cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
    if ptxas_v:
        cmd += ["-Xptxas", "-v"]
    _run(cmd, verbose)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False) -> None:
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    deps = _deps()
    if force or _stale(LIBBITMOE, srcs + deps):
        objs = []
        with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
            futs = []
            for s in srcs:
                o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
                objs.append(o)
                if force or _stale(o, [s] + deps):
                    futs.append(ex.submit(_compile, s, o, verbose, ptxas_v))
            for f in futs:
                f.result()
        tmp = LIBBITMOE + f".tmp{os.getpid()}"
        _run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
              *objs, "-o", tmp], verbose)
        os.replace(tmp, LIBBITMOE)
    ssrc = os.path.join(ROOT, "synth", "synth_dev.cu")
    if force or _stale(LIBSYNTH, [ssrc]):
        tmp = LIBSYNTH + f".tmp{os.getpid()}"
        _run([NVCC, *ARCH, *FLAGS, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
              ssrc, "-o", tmp], verbose)
        os.replace(tmp, LIBSYNTH)


if __name__ == "__main__":
    build(force="-f" in sys.argv, verbose="-v" in sys.argv, ptxas_v="--ptxas" in sys.argv)
