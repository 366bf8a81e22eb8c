"""Builds libmoe.so (the CUDA library behind include/moe.h) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
``sparse_moe_router_gb300/libmoe.so``.  The CUDA runtime is linked statically; the driver is
reached through the runtime's entry-point query (no -lcuda).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libmoe.so")
BUILD = os.path.join(ROOT, "_build")
# The same sources with MOE_DEBUG: every kernel checks the indices it reads from device data.
OUT_DEBUG = os.path.join(HERE, "libmoe_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "moe.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(out=OUT):
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force=False, verbose=False, extra=(), debug=False):
    """Compile the library if needed; returns the path of libmoe.so (debug=True: libmoe_debug.so,
    built with MOE_DEBUG)."""
    out = OUT_DEBUG if debug else OUT
    if not force and up_to_date(out):
        return out
    nvcc = _nvcc()
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(bdir, exist_ok=True)
    if debug:
        extra = tuple(extra) + ("-DMOE_DEBUG",)
    objs = []
    cmds = []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmds.append([nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=min(8, len(cmds))) as ex:
        for cmd, r in ex.map(run, cmds):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed for " + cmd[-3])
    tmp = out + ".tmp%d" % os.getpid()
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(link) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else (), debug="--debug" in sys.argv))
