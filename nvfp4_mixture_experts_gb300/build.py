"""Builds libnvfp4moe.so in-tree for sm_103a (one nvcc per translation unit, in parallel)."""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libnvfp4moe.so")
# the MOE_DEBUG flavour: bounds checks on every index read from a buffer (a bad one sets
# MOE_DEV_BAD_INDEX and its access is skipped); same symbols, separate file
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libnvfp4moe_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(os.path.dirname(HERE), "include", "nvfp4moe.h"), __file__]


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force=False, verbose=False, debug=False):
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []
    if debug:
        extra.append("-DMOE_DEBUG")

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [NVCC, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(len(_sources())) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + ".%d.tmp" % os.getpid()
    r = subprocess.run([NVCC, *FLAGS, "-shared", *objs, "-ldl", "-o", tmp], capture_output=True,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


def build_all(force=False):
    """Both flavours, side by side."""
    with ThreadPoolExecutor(2) as ex:
        return list(ex.map(lambda d: build(force=force, debug=d), (False, True)))


if __name__ == "__main__":
    if "--debug" in sys.argv:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug=True))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
