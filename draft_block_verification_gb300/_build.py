"""Build libsv.so in-tree: one nvcc job per translation unit (in parallel),
sm_103a only, then a shared-library link with the static CUDA runtime."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(HERE, "_lib")
LIBPATH = os.path.join(LIBDIR, "libsv.so")
SOURCES = ["sv_pass.cu", "sv_post.cu", "sv_api.cu", "sv_selftest.cu", "sv_static.cu",
           "sv_topk.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA 12.9+ with sm_103a support is required)")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "sv.h")]
    return max(os.path.getmtime(p) for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library if any source is newer than the built .so."""
    os.makedirs(LIBDIR, exist_ok=True)
    if not force and os.path.exists(LIBPATH) and os.path.getmtime(LIBPATH) >= _inputs():
        return LIBPATH
    nvcc = _nvcc()
    objs = [os.path.join(LIBDIR, f.replace(".cu", ".o")) for f in SOURCES]

    def one(src, obj):
        cmd = [nvcc] + ARCH + FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose:
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        list(ex.map(lambda a: one(*a), zip(SOURCES, objs)))
    tmp = LIBPATH + ".%d.tmp" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIBPATH)
    return LIBPATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
