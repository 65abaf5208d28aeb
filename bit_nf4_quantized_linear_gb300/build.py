"""Builds the in-tree CUDA library ``libnf4.so`` (sm_103a only) with nvcc, and
its checked debug variant ``libnf4_checked.so`` (``-DNF4_CHECKED=1``: in-kernel
index checks that record NF4_ERR_BOUNDS instead of accessing out of range; the
binding loads it when ``NF4_CHECKED=1`` is set in the environment).

The translation units compile in parallel; nothing is installed outside the
package directory.  ``python -m bit_nf4_quantized_linear_gb300.build`` or
``__graft_entry__.build()`` runs it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libnf4.so")
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libnf4_checked.so")
SOURCES = ["nf4_api.cu", "nf4_gemm.cu", "nf4_gemm8.cu", "nf4_gemm_f16.cu", "nf4_gemv.cu", "nf4_moe.cu", "nf4_quant.cu",
           "nf4_skinny.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                   "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC, *extra]


def _inputs_newer(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "nf4.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool = False) -> str:
    """Compile (when sources changed) and return the path of libnf4.so, or of
    libnf4_checked.so when `checked`."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    if not force and not _inputs_newer(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DNF4_CHECKED=1"] if checked else [])

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc(), *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_all(force: bool = False) -> list:
    """Both libraries, the normal and the checked build, compiled side by side."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda c: build(force=force, checked=c), (False, True)))


if __name__ == "__main__":
    if "--checked" in sys.argv:
        print(build(force="--force" in sys.argv, verbose=True, checked=True))
    else:
        print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
