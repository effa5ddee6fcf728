"""Builds the in-tree CUDA library ``_build/libpkv.so`` for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel (nvcc for
``.cu``, g++ for ``.cpp``) and linked into one shared library with the CUDA
runtime linked statically.  Run ``python -m paged_kv_decode_10_gb300.build``
or call :func:`build`.  Set ``PKV_PTXAS_VERBOSE=1`` to print register and
shared-memory use of every kernel.
"""
import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _sources():
    srcs = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))
    return [os.path.join(CSRC, f) for f in srcs]


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pkv.h")]


def _compile(src, verbose):
    obj = os.path.join(BUILD, "obj", os.path.basename(src) + ".o")
    if src.endswith(".cu"):
        cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            cmd[1:1] = ["-Xptxas", "-v"]
    else:
        cmd = ["g++", "-O2", "-fPIC", "-std=c++17", "-Wall", "-I", INCLUDE,
               "-I", "/usr/local/cuda/include", "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return obj, (res.stdout + res.stderr) if verbose else ""


def _fresh():
    if not os.path.exists(LIB):
        return False
    return os.path.getmtime(LIB) >= max(os.path.getmtime(p) for p in _deps())


def build(force=False, verbose=None):
    """Compile and link the library; returns its path.  Processes that build at
    the same time (one per rank) take turns on a lock file; a process that
    finds the library fresh once it holds the lock does nothing."""
    if verbose is None:
        verbose = os.environ.get("PKV_PTXAS_VERBOSE") == "1"
    os.makedirs(os.path.join(BUILD, "obj"), exist_ok=True)
    if not force and _fresh():
        return LIB
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and _fresh():
            return LIB
        return _build_locked(verbose)


def _build_locked(verbose):
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), srcs))
    if verbose:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = f"{LIB}.tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
