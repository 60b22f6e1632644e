"""Build libw4a16.so in place: nvcc for sm_103a, one object per translation unit, compiled in parallel.

Run as ``python -m w4a16_int4_weight_group_gb300.build`` or call ``build()``. Objects go to
``_build/`` next to this file; the shared library is written beside this file. The build is skipped
when the library is newer than every source and header.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import sysconfig
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libw4a16.so")

SOURCES = ["api.cu", "pack.cu", "gemm_generic.cu", "gemm_decode.cu", "gemm_prefill.cu"]
# CPython argument marshalling for the prepared-layer call (optional: the binding uses ctypes when it
# cannot be built, e.g. without the Python headers)
PYCALL_SRC = os.path.join(CSRC, "pycall.c")
PYCALL_PATH = os.path.join(HERE, "_w4a16_call" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "-I", INCLUDE, "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libw4a16.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h", ".c"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build_pycall(force: bool = False) -> bool:
    """Compile the CPython marshalling module beside the library; False when it cannot be built."""
    if not force and os.path.exists(PYCALL_PATH) and os.path.getmtime(PYCALL_PATH) >= os.path.getmtime(PYCALL_SRC):
        return True
    inc = sysconfig.get_paths().get("include")
    if not inc or not os.path.exists(os.path.join(inc, "Python.h")):
        return False
    cc = shutil.which(os.environ.get("CC", "cc")) or shutil.which("gcc")
    if not cc:
        return False
    tmp = PYCALL_PATH + ".tmp"
    r = subprocess.run([cc, "-O2", "-shared", "-fPIC", "-I", inc, PYCALL_SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        return False
    os.replace(tmp, PYCALL_PATH)
    return True


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    """Compile and link libw4a16.so (sm_103a) and the marshalling module. Returns the library path."""
    build_pycall(force)
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    jobs = jobs or min(len(SOURCES), os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
