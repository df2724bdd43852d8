"""Build the router's CUDA library in place, for sm_103a only.

Each .cu file under csrc/ compiles to an object in parallel (one -gencode),
then nvcc links them into lib/libmoe_router.so.  A rebuild happens only when a
source or header is newer than the library.

    python -m score_top_expert_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys
import sysconfig

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmoe_router.so")
# CPython entry points of the hot calls (argument conversion only), built
# where the interpreter's headers are installed
PYCALLS_SRC = os.path.join(CSRC, "pycalls.c")
PYCALLS = os.path.join(LIBDIR, "_pycalls" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}", f"-I{CSRC}"] + ARCH


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the router library needs the CUDA toolkit")


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [PYCALLS_SRC] +
            glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _python_include() -> str | None:
    inc = sysconfig.get_paths().get("include")
    return inc if inc and os.path.exists(os.path.join(inc, "Python.h")) else None


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    if not all(os.path.getmtime(p) <= t for p in _inputs()):
        return False
    if _python_include() is not None:
        return os.path.exists(PYCALLS) and os.path.getmtime(PYCALLS) >= t
    return True


def _build_pycalls() -> None:
    """The CPython call shim, linked against the library (found next to it)."""
    inc = _python_include()
    if inc is None:
        return
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        return
    tmp = PYCALLS + ".tmp"
    cmd = [cc, "-O2", "-shared", "-fPIC", f"-I{inc}", f"-I{INCLUDE}", PYCALLS_SRC,
           f"-L{LIBDIR}", "-lmoe_router", "-Wl,-rpath,$ORIGIN", "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the CPython call shim failed:\n{r.stderr}")
    os.replace(tmp, PYCALLS)


def _compile(src: str, verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + ["-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    """Compile and link the library; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = _sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), "-shared"] + ARCH + ["-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    _build_pycalls()
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
