"""Builds ``libmclayer.so`` in-tree for sm_103a with nvcc.

Every ``csrc/*.cu`` file is compiled to an object in parallel, then linked
into one shared library next to this file.  Run ``python -m
megatron_transformer_layer_gb300.build`` (or ``build()``).  ``build(debug=True)``
builds ``libmclayer_debug.so`` from the same sources with ``-DMC_DEBUG``: its
kernels check the indices of every global store against their extents and
record MC_ERR_DEVICE_BOUNDS instead of storing out of range (the binding
loads it when MC_LAYER_DEBUG=1 is set).  Both are compiled with
``-DMC_NVTX``: the layer's calls open one NVTX range per stage (F1..F7,
B1..B7, nested in ``mc_layer_forward`` / ``mc_layer_backward``), which a
profiler can show or filter on (``ncu --nvtx --nvtx-include ...``);
``build(nvtx=False)`` leaves them out.  NVTX v3 is header-only and costs a
pointer test per range when no tool is attached.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libmclayer.so")
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libmclayer_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libmclayer.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _compile(nvcc: str, src: str, extra: list[str], build_dir: str) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build(verbose: bool = False, extra_flags: list[str] | None = None, debug: bool = False,
          nvtx: bool = True) -> str:
    """Compile and link the library (the debug variant with `debug`);
    returns its path."""
    nvcc = _nvcc()
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    extra = list(extra_flags or []) + (["-DMC_DEBUG"] if debug else []) + \
        (["-DMC_NVTX"] if nvtx else [])
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, extra, build_dir), srcs))
    libdir = _cuda_lib_dir(nvcc)
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{libdir}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    if verbose:
        print(f"built {lib_path}")
    return lib_path


if __name__ == "__main__":
    args = [a for a in sys.argv[1:] if a != "--debug"]
    build(verbose=True, extra_flags=args, debug="--debug" in sys.argv[1:])
