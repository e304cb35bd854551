"""Build (nvcc, sm_103a) and load the TriMul C-ABI library ``libtrimul.so``.

The library is built in-tree under ``co_folding_pair_gb300/_build/``.  One
nvcc process per translation unit runs in parallel, then one link step; the
build is skipped when the library is newer than every source file.
"""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD, "libtrimul.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I" + INCLUDE]

_lock = threading.Lock()
_lib = None


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the TriMul CUDA library cannot be built")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "trimul.h"))
    return files


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every .cu under csrc/ for sm_103a and link libtrimul.so. Returns its path."""
    with _lock:
        if not force and not needs_build():
            return LIB_PATH
        os.makedirs(BUILD, exist_ok=True)
        nvcc = _nvcc()
        srcs = _sources()

        def compile_one(src):
            obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
            cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr)
            return obj

        with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
            objs = list(ex.map(compile_one, srcs))
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
        return LIB_PATH


class TrimulParams(ctypes.Structure):
    _fields_ = [
        ("D", ctypes.c_int),
        ("C", ctypes.c_int),
        ("W_a", ctypes.c_void_p),
        ("W_ga", ctypes.c_void_p),
        ("W_b", ctypes.c_void_p),
        ("W_gb", ctypes.c_void_p),
        ("W_o", ctypes.c_void_p),
        ("W_g", ctypes.c_void_p),
        ("ln_in_gamma", ctypes.c_void_p),
        ("ln_in_beta", ctypes.c_void_p),
        ("ln_out_gamma", ctypes.c_void_p),
        ("ln_out_beta", ctypes.c_void_p),
        ("eps", ctypes.c_float),
    ]


GRAD_FIELDS = ("dW_a", "dW_ga", "dW_b", "dW_gb", "dW_o", "dW_g",
               "d_ln_in_gamma", "d_ln_in_beta", "d_ln_out_gamma", "d_ln_out_beta")


class TrimulGrads(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in GRAD_FIELDS]


# Exported entry points: name -> (restype, argtypes).  Mirrors include/trimul.h.
_VP, _I, _U = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
SIGNATURES = {
    "trimul_create": (_I, [ctypes.POINTER(_VP), ctypes.POINTER(TrimulParams), _I]),
    "trimul_prepare": (_I, [_VP, _I, _I, _I]),
    "trimul_forward": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP, _VP, _U]),
    "trimul_forward_host": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP, _VP, _U]),
    "trimul_forward_noalloc": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP, _VP, _U]),
    "trimul_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "trimul_x_scale_log2": (_I, [_VP, _I]),
    "trimul_inproj": (_I, [_VP, _VP, _VP, _I, _I, _VP, _VP, _VP, _U]),
    "trimul_triangle": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP, _VP, _U]),
    "trimul_outproj": (_I, [_VP, _VP, _VP, _I, _I, _VP, _VP, _U]),
    "trimul_set_stage_events": (_I, [_VP, ctypes.POINTER(_VP)]),
    "trimul_destroy": (_I, [_VP]),
    "trimul_last_error": (ctypes.c_char_p, []),
    "trimul_kernels_per_forward": (_I, [_VP, _I, _I]),
    "trimul_kernels_per_forward_host": (_I, [_VP, _I, _I]),
    "trimul_host_join": (_I, [_VP, _VP]),
    "trimul_backward": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _VP, ctypes.POINTER(TrimulGrads), _VP, _U]),
    "trimul_backward_workspace_bytes": (ctypes.c_size_t, [_VP, _I, _I]),
    "trimul_kernels_per_backward": (_I, [_VP, _I, _I]),
}


def load(build_if_needed: bool = True):
    """Return the loaded ctypes library (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_needed:
        build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build the TriMul CUDA library first")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
