"""Build of the native library libcoll.so (nvcc, sm_103a, in-tree).

Every translation unit compiles in parallel; the link uses nvcc's default
static CUDA runtime so the library has no run-time path dependency beyond the
driver.  The result sits next to this file and is loaded by the package.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libcoll.so")

SOURCES = ["kernels.cu", "api.cpp", "derive.cpp", "static_ws.cu", "moe.cu", "composed.cu",
           "column.cu", "atom.cu"]
HEADERS = ["plan.h", "derive.h", "launch.h", "dev_common.cuh", "ll8.cuh", "ll128.cuh",
           "pipe.cuh", "sent.cuh", "policy_table.h", "tma.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No fast math: IEEE division/sqrt, no flush-to-zero (the fold is bit-exact).
COMMON = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo",
          "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
          "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")
    return path


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "coll.h"))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [cc, *COMMON]
        if src.endswith(".cu"):
            cmd += ARCH
        cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-shared", *ARCH, "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB
