"""Build libmha.so in-tree with nvcc for sm_103a (GB300).

Translation units compile in parallel into ``_build/`` and link into ``libmha.so`` next to
this file.  The CUDA runtime is linked statically; the driver is reached at run time
through ``cudaGetDriverEntryPointByVersion``, so no libcuda is needed at link time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libmha.so")
# the same library with the kernels' index checks compiled in (-DMHA_DEBUG_BOUNDS)
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libmha_debug.so")

SOURCES = ["capi.cu", "gemm_bf16.cu", "gemm_f32.cu", "sdpa_bf16.cu", "sdpa_f32.cu",
           "sdpa_decode.cu", "sdpa_bwd_f32.cu", "sdpa_bwd_bf16.cu", "bwd_util.cu", "layernorm.cu",
           "gemm_ln_bf16.cu", "gemm2_bf16.cu",
           "layer_noalloc.cu", "layer_host.cu"]
HEADERS = ["device_common.cuh", "launchers.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libmha.so")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "mha.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug_bounds: bool = False) -> str:
    """Compile every translation unit and link libmha.so (libmha_debug.so, the kernels' index
    checks compiled in, with debug_bounds); returns the library path."""
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug_bounds else BUILD_DIR
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + NVCC_FLAGS + list(extra_flags or [])
    if debug_bounds:
        flags.append("-DMHA_DEBUG_BOUNDS")

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
