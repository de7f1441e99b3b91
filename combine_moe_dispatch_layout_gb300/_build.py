"""Build ``libmoe_ep.so`` for sm_103a with nvcc (in-tree, no cmake).

Each ``csrc/*.cu`` translation unit compiles in parallel to an object under
``_build/``; the objects link into ``libmoe_ep.so`` next to this file.  The
flags keep IEEE semantics everywhere the pipeline does floating point: no
fast-math, no FMA contraction (``-fmad=false``), IEEE division and square
root, no flush-to-zero.  ``-Xptxas -v`` reports (registers, spills, shared
memory) go to ``_build/<unit>.ptxas.txt``.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_ep.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
    "-fmad=false", "--prec-div=true", "--prec-sqrt=true", "-ftz=false",
    "-I" + INCLUDE, "-I" + CSRC, "-Xptxas", "-v",
]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__])


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(nvcc, src):
    name = os.path.splitext(os.path.basename(src))[0]
    obj = os.path.join(BUILD, name + ".o")
    log = os.path.join(BUILD, name + ".ptxas.txt")
    r = subprocess.run([nvcc, *NVCC_FLAGS, "-c", src, "-o", obj],
                       capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stderr[-4000:]))
    return obj


def build(force=False):
    """Compile every translation unit and link libmoe_ep.so; returns its path."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s), srcs))
    tmp = LIB + ".%d.tmp" % os.getpid()
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv))
