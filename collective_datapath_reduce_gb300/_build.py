"""Build the C-ABI library libpurlin_gb.so from csrc/ with nvcc (sm_103a only).

Translation units compile in parallel into _build/ next to this file; the
shared library lands in lib/.  Nothing is rebuilt when every object is newer
than the sources and headers.  Host code is plain C++17 (no intrinsics, no
-march), so the same sources build on x86_64 and aarch64 hosts.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIBNAME = "libpurlin_gb.so"
LIBPATH = os.path.join(LIBDIR, LIBNAME)
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIBPATH_DEBUG = os.path.join(LIBDIR, "libpurlin_gb_debug.so")
EXAMPLES = os.path.join(PKG, "examples")
EXAMPLES_PATH = os.path.join(LIBDIR, "libpurlin_examples.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE binary32 arithmetic throughout: no flush-to-zero, no contraction, exact division.
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
          "-fmad=false", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libpurlin_gb.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.cuh")))


def _newest(paths):
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def build_examples(verbose: bool = False, force: bool = False) -> str:
    """Compile (if needed) the device-side API examples into libpurlin_examples.so.

    They use only the public headers (include/purlin_device.cuh and
    include/purlin_atoms.cuh), as a user's own kernels would."""
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(EXAMPLES, "*.cu")))
    newest = max(_newest(srcs), _newest(glob.glob(os.path.join(INCLUDE, "*.cuh"))))
    if not force and os.path.exists(EXAMPLES_PATH) and os.path.getmtime(EXAMPLES_PATH) >= newest:
        return EXAMPLES_PATH
    tmp = EXAMPLES_PATH + ".tmp"
    cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
           "-fmad=false", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-shared", *srcs, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, EXAMPLES_PATH)
    return EXAMPLES_PATH


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile (if needed) and return the path of libpurlin_gb.so (and the examples library).

    debug=True builds the checking library libpurlin_gb_debug.so instead
    (PURLIN_DEBUG: every kernel checks each work item against the rank
    buffers' sizes before it moves data)."""
    bdir = BUILD_DEBUG if debug else BUILD
    libpath = LIBPATH_DEBUG if debug else LIBPATH
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = _sources()
    hdr_time = _newest(_headers())
    cc = nvcc()
    jobs = []
    objs = []
    for src in srcs:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_time):
            cmd = [cc, *ARCH, *CFLAGS, *(["-DPURLIN_DEBUG"] if debug else []), "-c", src, "-o", obj]
            if src.endswith(".cu") and verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose and (r.stdout or r.stderr):
                    print(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if jobs or not os.path.exists(libpath) or os.path.getmtime(libpath) < _newest(objs):
        tmp = libpath + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        os.replace(tmp, libpath)
    if not debug:
        build_examples(verbose, force)
    return libpath


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
