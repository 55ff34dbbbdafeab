"""Build librope.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file is compiled in parallel to an object, then linked
into ``lib/librope.so`` with the CUDA runtime linked statically (the library
then loads on hosts without a GPU, and uses the caller's CUDA context and
streams on hosts with one).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import uuid
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIBRARY = os.path.join(LIBDIR, "librope.so")
OBJDIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librope")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "rope.h")]


def up_to_date(output: str = LIBRARY) -> bool:
    if not os.path.exists(output):
        return False
    t = os.path.getmtime(output)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, extra_flags: list[str] | None = None, output: str = LIBRARY,
          verbose: bool = False) -> str:
    """Compile every .cu under csrc/ and link ``output``; returns its path."""
    if not force and not extra_flags and up_to_date(output):
        return output
    os.makedirs(OBJDIR, exist_ok=True)
    os.makedirs(os.path.dirname(output), exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + ARCH + list(extra_flags or [])
    tag = "%d_%s" % (os.getpid(), uuid.uuid4().hex[:8])   # unique per build, even in one process

    def compile_one(src):
        obj = os.path.join(OBJDIR, os.path.basename(src) + "." + tag + ".o")
        p = subprocess.run([cc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, p.stdout, p.stderr))
        return obj, p.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = output + "." + tag
    p = subprocess.run([cc, "-shared", "-cudart", "static", *ARCH, "-o", tmp, *objs],
                       capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (p.stdout, p.stderr))
    os.replace(tmp, output)
    for o in objs:
        os.remove(o)
    return output


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
