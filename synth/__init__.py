"""Seeded synthetic inputs, shared by the oracle side and the CUDA side.

This module only turns seeds into numbers (see ``synth.c`` for the exact
definitions); it holds none of the paged-attention arithmetic.  The
workload recipes in :mod:`synth.workloads` describe the shapes of the
workloads on the PagedAttention pages (skewed length mix, 16-token blocks,
shared prefixes, 128K contexts) and which stream feeds which tensor.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (plain gcc, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_u64.restype = u64
            lib.synth_u64.argtypes = [u64, u64]
            lib.synth_stream_seed.restype = u64
            lib.synth_stream_seed.argtypes = [u64, u64]
            lib.synth_uniform.restype = f64
            lib.synth_uniform.argtypes = [u64, u64]
            lib.synth_uniform_int.restype = i64
            lib.synth_uniform_int.argtypes = [u64, u64, i64, i64]
            for name in ("synth_fill_normal_f32", "synth_fill_normal_bf16", "synth_fill_normal_f64"):
                fn = getattr(lib, name)
                fn.restype = None
                fn.argtypes = [u64, u64, u64, vp, f64]
            lib.synth_fill_uniform_int.restype = None
            lib.synth_fill_uniform_int.argtypes = [u64, u64, u64, i64, i64, vp]
            lib.synth_lengths_mix.restype = None
            lib.synth_lengths_mix.argtypes = [u64, u64, vp]
            lib.synth_permutation.restype = None
            lib.synth_permutation.argtypes = [u64, i32, vp]
            _lib = lib
    return _lib


M64 = (1 << 64) - 1


def u64(seed: int, counter: int) -> int:
    return int(_load().synth_u64(seed & M64, counter & M64))


def stream_seed(base: int, tag: int) -> int:
    return int(_load().synth_stream_seed(base & M64, tag & M64))


def uniform(seed: int, counter: int) -> float:
    return float(_load().synth_uniform(seed & M64, counter & M64))


def uniform_int(seed: int, counter: int, lo: int, hi: int) -> int:
    return int(_load().synth_uniform_int(seed & M64, counter & M64, lo, hi))


def normal(seed: int, n: int, dtype: str = "f32", offset: int = 0, scale: float = 1.0) -> np.ndarray:
    """Elements ``offset .. offset+n-1`` of the N(0,1)*scale stream ``seed``.

    ``dtype`` is ``"f32"`` (float32), ``"bf16"`` (uint16 bf16 bit patterns,
    RNE from the fp32 value) or ``"f64"``.
    """
    lib = _load()
    if dtype == "f32":
        out = np.empty(n, np.float32)
        lib.synth_fill_normal_f32(seed & M64, offset, n, out.ctypes.data, scale)
    elif dtype == "bf16":
        out = np.empty(n, np.uint16)
        lib.synth_fill_normal_bf16(seed & M64, offset, n, out.ctypes.data, scale)
    elif dtype == "f64":
        out = np.empty(n, np.float64)
        lib.synth_fill_normal_f64(seed & M64, offset, n, out.ctypes.data, scale)
    else:
        raise ValueError(dtype)
    return out


def uniform_ints(seed: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_fill_uniform_int(seed & M64, offset, n, lo, hi, out.ctypes.data)
    return out


def lengths_mix(seed: int, n: int) -> np.ndarray:
    """n lengths from the 70 % U[32,511] / 25 % U[512,2047] / 5 % U[2048,4095] mix."""
    out = np.empty(n, np.int32)
    _load().synth_lengths_mix(seed & M64, n, out.ctypes.data)
    return out


def permutation(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_permutation(seed & M64, n, out.ctypes.data)
    return out

