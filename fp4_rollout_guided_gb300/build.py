"""Builds libtrace_fp4.so in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link into one shared library
under ``fp4_rollout_guided_gb300/_build``.  Flags: -O3, no fused multiply-add
contraction (-fmad=false), IEEE division/square root and no flush-to-zero
(nvcc's defaults, stated explicitly), line info for the profiler.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libtrace_fp4.so")
SOURCES = ["trace_kernels.cu", "trace_fakequant.cu", "trace_gemm.cu", "trace_gemm_tc.cu",
           "trace_api.cu", "trace_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-prec-div=true",
              "-prec-sqrt=true", "-ftz=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libtrace_fp4.so")
    return path


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
              if f.endswith((".h", ".cuh"))]
    files.append(os.path.join(INCLUDE, "trace_fp4.h"))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_dir: str = None) -> str:
    """Builds the library; `extra_flags` / `out_dir` build a variant elsewhere."""
    out = out_dir or BUILD
    lib_path = os.path.join(out, "libtrace_fp4.so")
    if out_dir is None and not force and not stale():
        return LIB
    os.makedirs(out, exist_ok=True)
    cc = nvcc()

    # where the NVFP4 GEMM looks for cuBLASLt if the loader's search fails
    lib_dir = os.path.realpath(os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(cc))),
                                            "lib64"))

    def compile_one(src):
        obj = os.path.join(out, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, f'-DTRACE_CUDA_LIB_DIR="{lib_dir}"', *extra_flags, "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib_path + f".{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
