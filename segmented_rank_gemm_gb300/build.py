"""Build the layer's CUDA library in-tree: ``segmented_rank_gemm_gb300/liblora_layer.so``.

Each ``csrc/*.cu`` file is compiled by nvcc for sm_103a only (in parallel), then linked
into one shared library with the C ABI of ``include/lora_layer.h``.  Run as
``python -m segmented_rank_gemm_gb300.build`` or through ``__graft_entry__.build()``.

``build(debug=True)`` (``--debug``) builds the debug flavour, ``liblora_layer_debug.so``,
compiled with ``-DLORA_DEBUG``: the kernels check the indices they take from data (slot rows
of the adapter pools, rows of the delta and v buffers, K-split planes) and, instead of
accessing memory outside a buffer, skip the access and raise a device flag that
``lora_get_status`` reports as LORA_EBOUNDS.  The binding loads it when the environment
variable ``LORA_LAYER_LIBRARY`` is ``debug``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "liblora_layer.so")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "liblora_layer_debug.so")


def library_path() -> str:
    """The flavour the binding loads: the debug one if LORA_LAYER_LIBRARY=debug."""
    flavour = os.environ.get("LORA_LAYER_LIBRARY", "")
    if flavour not in ("", "release", "debug"):
        raise ValueError("LORA_LAYER_LIBRARY must be 'release' or 'debug', not %r" % flavour)
    return DEBUG_LIB_PATH if flavour == "debug" else LIB_PATH

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the layer")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "lora_layer.h"),
                                      os.path.abspath(__file__)]


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if debug:
        extra_flags = ("-DLORA_DEBUG", *extra_flags)
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nv = nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nv, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".%d.tmp" % os.getpid()
    cmd = [nv, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-lpthread", "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
