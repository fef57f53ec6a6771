"""Builds the in-tree CUDA library ``_build/libretention.so`` for sm_103a.

Plain nvcc, one object per ``csrc/*.cu`` compiled in parallel, then one
shared-library link.  Objects are rebuilt when their source or any header
is newer.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libretention.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
# RET_NVTX=1: an NVTX range around each ABI call (build with force=True when
# switching, since objects are only rebuilt when sources change).
if os.environ.get("RET_NVTX") == "1":
    NVCC_FLAGS = NVCC_FLAGS + ["-DRET_NVTX"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _newest_header():
    hdrs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max((os.path.getmtime(h) for h in hdrs), default=0.0)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(os.path.join(BUILD, "obj"), exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _newest_header()
    nvcc = _nvcc()

    def obj_of(s):
        return os.path.join(BUILD, "obj", os.path.basename(s)[:-3] + ".o")

    def compile_one(s):
        o = obj_of(s)
        if (not force and os.path.exists(o)
                and os.path.getmtime(o) >= max(os.path.getmtime(s), hdr_t)):
            return o, None
        cmd = [nvcc] + NVCC_FLAGS + ["-c", s, "-o", o + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            return o, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
        os.replace(o + ".tmp", o)
        return o, (r.stderr if verbose and r.stderr else None)

    with cf.ThreadPoolExecutor(max_workers=min(16, len(srcs) or 1)) as ex:
        results = list(ex.map(compile_one, srcs))
    errs = [e for _, e in results if e and "error" in e.lower()]
    if errs:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errs))
    objs = [o for o, _ in results]
    if (force or not os.path.exists(LIB)
            or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs)):
        cmd = [nvcc] + ARCH + ["-shared", "-o", LIB + ".tmp"] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
