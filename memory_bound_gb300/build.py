"""Build libmemory_bound.so (CUDA for sm_103a) in-tree.

Each translation unit under csrc/ is compiled by nvcc in parallel, then the
objects are linked into memory_bound_gb300/libmemory_bound.so with the CUDA
runtime linked statically (the library needs only the driver at run time).
"""
import glob
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmemory_bound.so")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
         "-I", INCLUDE, "-I", CSRC]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    deps = (glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])          # flags and arch live here
    return all(os.path.getmtime(p) <= t for p in deps)


def _compile(src, objdir, verbose):
    obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
    return obj, res.stderr


def build(force=False, verbose=False):
    """Compile every CUDA source and link the shared library; return its path."""
    if not force and _up_to_date():
        return LIB
    # Objects go to a directory of this process's own and the library is
    # linked to a file of its own, then renamed over the old one, so builds
    # started at once by several processes never read each other's halves.
    os.makedirs(OBJDIR, exist_ok=True)
    objdir = tempfile.mkdtemp(prefix="objs-", dir=OBJDIR)
    tmp = f"{LIB}.tmp{os.getpid()}"
    try:
        srcs = _sources()
        with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
            results = list(ex.map(lambda s: _compile(s, objdir, verbose), srcs))
        if verbose:
            for _, log in results:
                sys.stderr.write(log)
        objs = [o for o, _ in results]
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + res.stderr)
        os.replace(tmp, LIB)
    finally:
        shutil.rmtree(objdir, ignore_errors=True)
        if os.path.exists(tmp):
            os.remove(tmp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
