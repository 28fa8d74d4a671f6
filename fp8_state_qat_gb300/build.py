"""Compile the CUDA library ``libgdnqat.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel (one ``-gencode``, no cmake), then
linked into ``fp8_state_qat_gb300/_lib/libgdnqat.so`` with the CUDA runtime linked
statically. Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libgdnqat.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return p


def _sources(csrc=CSRC):
    return sorted(glob.glob(os.path.join(csrc, "*.cu")))


def headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + [
        os.path.join(ROOT, "include", "gdnqat.h"), __file__]


def _deps():
    return _sources() + headers()


def newer_than(out: str, deps) -> bool:
    """`out` exists and no file in `deps` was modified after it."""
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(d) <= t for d in deps)


def up_to_date() -> bool:
    return newer_than(LIB_PATH, _deps())


def compile_library(sources, out: str, obj_dir: str, verbose: bool = False) -> str:
    """nvcc each of `sources` (objects in `obj_dir`, in parallel) and link them into the shared
    library `out` with the CUDA runtime linked statically. A source is a path, or a pair
    (path, extra -D macros for that file)."""
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                    "-I", os.path.join(ROOT, "include")]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(item):
        src, defines = (item, ()) if isinstance(item, str) else item
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *flags, *[f"-D{d}" for d in defines], "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, sources))
    if verbose:
        for _, log in results:
            print(log)
    tmp = out + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu into libgdnqat.so (skipped when it is up to date)."""
    if not force and up_to_date():
        return LIB_PATH
    return compile_library(_sources(), LIB_PATH, OBJ_DIR, verbose=verbose)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
