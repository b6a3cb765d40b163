"""In-tree build of ``libmhc_gb300.so`` for sm_103a (GB300).

Each ``csrc/*.cu`` file is compiled by its own ``nvcc`` process (in parallel)
with ``-gencode arch=compute_103a,code=sm_103a``, then the objects are linked
into one shared library next to this file.  Only sources newer than their
object are recompiled.  Run ``python gemm_rms_sinkhorn_gb300/build.py``
(``--check``: the MHC_CHECK build, ``libmhc_gb300_check.so``, beside it).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmhc_gb300.so")
# the build with device index checks (-DMHC_CHECK): same sources, own objects
BUILD_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "libmhc_gb300_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE,
              "-I" + CSRC, "-Wno-deprecated-gpu-targets"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _compile(nvcc, src, obj, extra, verbose):
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, res.stdout, res.stderr))
    return res.stdout + res.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          check: bool = False) -> str:
    """Builds libmhc_gb300.so, or with check=True libmhc_gb300_check.so, whose
    kernels record a failed device index check instead of touching memory out
    of range (csrc/check.cuh)."""
    nvcc = _nvcc()
    build_dir, lib = (BUILD_CHECK, LIB_CHECK) if check else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_hdr = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if check:
        extra.append("-DMHC_CHECK")
    jobs = []
    objs = []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        stale = (force or ptxas_info or not os.path.exists(obj) or
                 os.path.getmtime(obj) < max(os.path.getmtime(src), newest_hdr))
        if stale:
            jobs.append((src, obj))
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            outs = list(ex.map(lambda j: _compile(nvcc, j[0], j[1], extra, verbose), jobs))
        if ptxas_info:
            for (src, _), out in zip(jobs, outs):
                print("== %s\n%s" % (os.path.basename(src), out))
    if jobs or not os.path.exists(lib) or os.path.getmtime(lib) < max(map(os.path.getmtime, objs)):
        tmp = lib + ".%d.tmp" % os.getpid()
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                check="--check" in sys.argv))
