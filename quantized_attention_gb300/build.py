"""Builds libqattn.so in-tree with nvcc for sm_103a (no CMake, no torch
extension machinery).  Translation units compile in parallel; the result lands
in ``quantized_attention_gb300/_lib/libqattn.so``, and the checked build
(``checked=True``: -DQATTN_CHECK=1, every kernel's computed indices guarded,
see include/qattn.h) in ``quantized_attention_gb300/_lib/check/libqattn.so``."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libqattn.so")
CHECK_DIR = os.path.join(OUT_DIR, "check")
CHECK_LIB = os.path.join(CHECK_DIR, "libqattn.so")
SOURCES = ["qattn_api.cu", "quant_kernels.cu", "attn_fwd.cu", "qattn_noalloc.cu", "decode.cu", "exact24.cu",
           "intsm.cu", "attn_short.cu", "peaks.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libqattn.so")


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")


def build(verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    out_dir = CHECK_DIR if checked else OUT_DIR
    lib_path = CHECK_LIB if checked else LIB
    if checked:
        extra_flags = (*extra_flags, "-DQATTN_CHECK=1")
    os.makedirs(out_dir, exist_ok=True)
    objs_dir = os.path.join(out_dir, "obj")
    os.makedirs(objs_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(objs_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "shared",
           "-Xlinker", "-rpath", "-Xlinker", cuda_lib_dir()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_all(verbose: bool = False) -> tuple[str, str]:
    """The normal and the checked library, compiled side by side."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        normal = ex.submit(build, verbose)
        chk = ex.submit(build, verbose, (), True)
        return normal.result(), chk.result()


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
