"""Builds libxqa.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each ``csrc/*.cu`` translation unit compiles in parallel to an object file
under ``_build/``; the objects link into ``paged_fp8_kv_gqa_gb300/libxqa.so``
with the CUDA runtime linked statically. A unit is rebuilt only when it or a
header is newer than its object. ``ptxas -v`` register/spill/shared-memory
reports are kept in ``_build/ptxas_<unit>.log``.

``build(variant="stamps")`` builds the diagnostic library
``_build/stamps/libxqa_stamps.so`` instead: the same sources compiled with
``-DXQA_STAMPS``, whose partial kernel also records per-CTA phase timestamps
(read back with ``xqa_diag_read_stamps``; used by ``bench.py --stamps``).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libxqa.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3",
    "-std=c++17",
    "-lineinfo",
    "-Xcompiler",
    "-fPIC",
    "-Xptxas",
    "-v",
    "-I",
    INCLUDE,
    "-I",
    CSRC,
]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libxqa.so")


def _newest_header() -> float:
    hdrs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    hdrs += glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hdrs), default=0.0)


VARIANTS = {"": [], "stamps": ["-DXQA_STAMPS"]}


def _paths(variant: str):
    """(build directory, library path) of a build variant."""
    if variant == "":
        return BUILD_DIR, LIB_PATH
    d = os.path.join(BUILD_DIR, variant)
    return d, os.path.join(d, f"libxqa_{variant}.so")


def _compile(nvcc: str, src: str, force: bool, variant: str = "") -> str:
    bdir, _ = _paths(variant)
    name = os.path.splitext(os.path.basename(src))[0]
    obj = os.path.join(bdir, name + ".o")
    if (not force and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(src), _newest_header())):
        return obj
    cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, *VARIANTS[variant], "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(bdir, f"ptxas_{name}.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    """Compile and link libxqa.so (or a diagnostic variant); returns its path."""
    nvcc = nvcc_path()
    bdir, lib_path = _paths(variant)
    os.makedirs(bdir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, force, variant), sources))
    newest_obj = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(lib_path) or os.path.getmtime(lib_path) < newest_obj:
        tmp = lib_path + ".tmp"
        cmd = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib_path)
    if verbose:
        for log in sorted(glob.glob(os.path.join(bdir, "ptxas_*.log"))):
            with open(log) as f:
                print(f.read())
    return lib_path


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                variant="stamps" if "--stamps" in sys.argv else ""))
