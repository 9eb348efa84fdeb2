"""Build librcu.so (the C-ABI CUDA library) for sm_103a with nvcc.

Each .cu file is compiled to an object in parallel, then linked into
``recurrent_cell_unroll_gb300/_lib/librcu.so`` with the static CUDA runtime.
Objects are rebuilt only when a source or header is newer.  ``build(debug=True)``
makes ``librcu_debug.so`` instead: the same sources with -DRCU_DEBUG, whose
kernels check their global-memory indices and record a failed check in the
device error word (RCU_ERR_CUDA from the status calls) instead of accessing.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "librcu.so")
LIB_DEBUG = os.path.join(LIBDIR, "librcu_debug.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags():
    return ["-O3", "-lineinfo", ARCH, "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
            "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _newest_header():
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def build(verbose: bool = False, jobs: int = 0, debug: bool = False) -> str:
    objdir = OBJDIR + ("_debug" if debug else "")
    lib = LIB_DEBUG if debug else LIB
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _newest_header()
    cmds = []
    objs = []
    for s in srcs:
        o = os.path.join(objdir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if os.path.exists(o) and os.path.getmtime(o) >= max(os.path.getmtime(s), hdr_t):
            continue
        cmds.append([nvcc(), *_flags(), *(["-DRCU_DEBUG"] if debug else []), "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return r

    if cmds:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(cmds), os.cpu_count() or 4)) as ex:
            list(ex.map(run, cmds))
    if cmds or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc(), ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static", "-lrt", "-ldl",
             "-lpthread"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
