"""ORACLE -- test infrastructure only.

A plain, slow, obviously correct CPU statement of the paged-attention hot
path, written from the PagedAttention pages.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with the CUDA library (``paged_kv_cache_280_gb300``)
and never imports it.

Parts:
  * ``pa_oracle.c``  -- fp64 decode attention (direct and split + reduce),
    paged prefill (chunked causal) attention, the slot-mapped append, the
    copy-on-write block copy, and the FP8 (E4M3) pool's codes, append and
    decode, as element loops over host arrays.
  * ``alloc_model``  -- a reference model of the block allocator
    (on-demand blocks, refcounted sharing, copy-on-write).
  * ``waste``        -- the memory accounting of the waste simulation on
    the ohmygp.com page (contiguous reservation vs paged blocks).

Inputs are numpy arrays: fp32 tensors as ``float32``, bf16 tensors as
``uint16`` bit patterns (widened exactly inside the C code).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {-1: "bad argument", -2: "block id out of range", -3: "slot out of range", -4: "out of memory"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile ``libpa_oracle.so`` next to its source (plain gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _open(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i32, f64, vp = ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
    lib.oracle_decode_attention.restype = ctypes.c_int
    lib.oracle_decode_attention.argtypes = [ctypes.c_int, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                            i32, i32, i32, f64, i32, i32, vp]
    lib.oracle_decode_partials.restype = ctypes.c_int
    lib.oracle_decode_partials.argtypes = [ctypes.c_int, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                           i32, i32, i32, f64, i32, i32, vp, vp, vp]
    lib.oracle_combine_partials.restype = ctypes.c_int
    lib.oracle_combine_partials.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    lib.oracle_reshape_and_cache.restype = ctypes.c_int
    lib.oracle_reshape_and_cache.argtypes = [i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32]
    lib.oracle_copy_blocks.restype = ctypes.c_int
    lib.oracle_copy_blocks.argtypes = [i32, vp, vp, vp, i32, i32, i32, i32, i32]
    lib.oracle_e4m3_encode_array.restype = None
    lib.oracle_e4m3_encode_array.argtypes = [vp, ctypes.c_int64, vp]
    lib.oracle_e4m3_value_array.restype = None
    lib.oracle_e4m3_value_array.argtypes = [vp, ctypes.c_int64, vp]
    lib.oracle_reshape_and_cache_fp8.restype = ctypes.c_int
    lib.oracle_reshape_and_cache_fp8.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                 ctypes.c_float, ctypes.c_float]
    lib.oracle_decode_attention_fp8.restype = ctypes.c_int
    lib.oracle_decode_attention_fp8.argtypes = [ctypes.c_int, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, i32,
                                                vp, i32, i32, i32, i32, i32, i32, f64, i32, i32, vp]
    lib.oracle_prefill_attention.restype = ctypes.c_int
    lib.oracle_prefill_attention.argtypes = [ctypes.c_int, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                             i32, i32, f64, i32, i32, vp]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build())
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"oracle error {rc}"))


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    raise TypeError(f"oracle tensors are float32 or uint16 (bf16 bits), got {a.dtype}")


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


def decode_attention(q, k_pool, v_pool, block_tables, seq_lens, scale, seqs=None, threads=1):
    """fp64 decode attention.  Returns out[B][Hq][D] (float64).

    q: [B][Hq][D]; pools: [num_blocks][Hkv][bs][D]; block_tables: [B][max_blocks] int32;
    seq_lens: [B] int32.  ``seqs`` restricts the computation to those sequence
    indices (other rows are NaN); ``threads`` > 1 runs sequences on a thread pool.
    """
    q, k_pool, v_pool = _c(q), _c(k_pool), _c(v_pool)
    dt = _dtype_code(q)
    if _dtype_code(k_pool) != dt or _dtype_code(v_pool) != dt:
        raise TypeError("q and the pools must share a dtype")
    bt = _c(block_tables, np.int32)
    lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    nb, Hkv, bs, D2 = k_pool.shape
    assert D2 == D and v_pool.shape == k_pool.shape and bt.shape[0] == B and lens.shape == (B,)
    out = np.full((B, Hq, D), np.nan, np.float64)
    lib = _load()
    todo = list(range(B)) if seqs is None else sorted(set(int(s) for s in seqs))

    def run(b):
        _check(lib.oracle_decode_attention(dt, q.ctypes.data, k_pool.ctypes.data, v_pool.ctypes.data,
                                           bt.ctypes.data, bt.shape[1], lens.ctypes.data, B, Hq, Hkv, D,
                                           bs, nb, float(scale), b, b + 1, out.ctypes.data))

    if threads <= 1:
        for b in todo:
            run(b)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, todo))
    return out


def prefill_attention(q, k_pool, v_pool, block_tables, seq_lens, cu_q_lens, scale, seqs=None, threads=1):
    """fp64 paged prefill (chunked causal) attention.  Returns out[T][Hq][D] (float64).

    q: [T][Hq][D] with T = cu_q_lens[-1]; chunk token i of sequence b is row
    cu_q_lens[b] + i at position seq_lens[b] - n_b + i, and sees keys 0..that
    position.  ``seqs`` restricts the computation to those sequences (other
    rows are NaN); ``threads`` > 1 runs sequences on a thread pool.
    """
    q, k_pool, v_pool = _c(q), _c(k_pool), _c(v_pool)
    dt = _dtype_code(q)
    if _dtype_code(k_pool) != dt or _dtype_code(v_pool) != dt:
        raise TypeError("q and the pools must share a dtype")
    bt = _c(block_tables, np.int32)
    lens = _c(seq_lens, np.int32)
    cu = _c(cu_q_lens, np.int32)
    T, Hq, D = q.shape
    nb, Hkv, bs, D2 = k_pool.shape
    B = lens.shape[0]
    assert D2 == D and v_pool.shape == k_pool.shape and bt.shape[0] == B and cu.shape == (B + 1,) and cu[-1] == T
    out = np.full((T, Hq, D), np.nan, np.float64)
    lib = _load()
    todo = list(range(B)) if seqs is None else sorted(set(int(s) for s in seqs))

    def run(b):
        _check(lib.oracle_prefill_attention(dt, q.ctypes.data, k_pool.ctypes.data, v_pool.ctypes.data,
                                            bt.ctypes.data, bt.shape[1], lens.ctypes.data, cu.ctypes.data, B, Hq,
                                            Hkv, D, bs, nb, float(scale), b, b + 1, out.ctypes.data))

    if threads <= 1:
        for b in todo:
            run(b)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, todo))
    return out


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> OCP FP8 E4M3 codes (nearest, ties to even mantissa, saturating at 448)."""
    x = _c(np.asarray(x, np.float32))
    out = np.empty(x.shape, np.uint8)
    _load().oracle_e4m3_encode_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def e4m3_value(codes) -> np.ndarray:
    """E4M3 codes -> their values (float64; the NaN code gives NaN)."""
    codes = _c(np.asarray(codes, np.uint8))
    out = np.empty(codes.shape, np.float64)
    _load().oracle_e4m3_value_array(codes.ctypes.data, codes.size, out.ctypes.data)
    return out


def reshape_and_cache_fp8(k_new, v_new, k_pool, v_pool, slot_mapping, k_scale, v_scale):
    """In-place slot-mapped append into FP8 pools (uint8 codes of x / scale)."""
    assert k_pool.dtype == np.uint8 and k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    k_new, v_new = _c(k_new), _c(v_new)
    slots = _c(slot_mapping, np.int64)
    nb, Hkv, bs, D = k_pool.shape
    _check(_load().oracle_reshape_and_cache_fp8(_dtype_code(k_new), k_new.ctypes.data, v_new.ctypes.data,
                                                k_pool.ctypes.data, v_pool.ctypes.data, slots.ctypes.data, len(slots),
                                                Hkv, D, bs, nb, float(k_scale), float(v_scale)))


def decode_attention_fp8(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, scale, seqs=None, threads=1):
    """fp64 decode attention over FP8 pools (K^ = value * k_scale, V^ = value * v_scale); out[B][Hq][D]."""
    q = _c(q)
    dt = _dtype_code(q)
    k_pool, v_pool = _c(k_pool, np.uint8), _c(v_pool, np.uint8)
    bt = _c(block_tables, np.int32)
    lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    nb, Hkv, bs, _ = k_pool.shape
    out = np.full((B, Hq, D), np.nan, np.float64)
    lib = _load()
    todo = list(range(B)) if seqs is None else sorted(set(int(s) for s in seqs))
    ranges = [(b, b + 1) for b in todo] if threads > 1 else [(min(todo), max(todo) + 1)] if todo else []

    def run(r):
        _check(lib.oracle_decode_attention_fp8(dt, q.ctypes.data, k_pool.ctypes.data, v_pool.ctypes.data,
                                               float(k_scale), float(v_scale), bt.ctypes.data, bt.shape[1],
                                               lens.ctypes.data, B, Hq, Hkv, D, bs, nb, float(scale), r[0], r[1],
                                               out.ctypes.data))

    if threads <= 1:
        for r in ranges:
            run(r)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, ranges))
    if seqs is not None:
        keep = np.zeros(B, bool)
        keep[todo] = True
        out[~keep] = np.nan
    return out


def decode_partials(q, k_pool, v_pool, block_tables, seq_lens, scale, partition_tokens):
    """Per-partition (m, l, o) of the split form; shapes [B][Hq][P], [B][Hq][P], [B][Hq][P][D]."""
    q, k_pool, v_pool = _c(q), _c(k_pool), _c(v_pool)
    dt = _dtype_code(q)
    bt = _c(block_tables, np.int32)
    lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    nb, Hkv, bs, _ = k_pool.shape
    n_part = max(1, int(-(-int(lens.max(initial=0)) // partition_tokens)))
    m = np.empty((B, Hq, n_part), np.float64)
    l = np.empty((B, Hq, n_part), np.float64)
    o = np.empty((B, Hq, n_part, D), np.float64)
    _check(_load().oracle_decode_partials(dt, q.ctypes.data, k_pool.ctypes.data, v_pool.ctypes.data,
                                          bt.ctypes.data, bt.shape[1], lens.ctypes.data, B, Hq, Hkv, D, bs,
                                          nb, float(scale), int(partition_tokens), n_part, m.ctypes.data,
                                          l.ctypes.data, o.ctypes.data))
    return m, l, o


def combine_partials(m, l, o):
    """The split-sequence reduce; returns out[..., D] (float64)."""
    m, l, o = _c(m, np.float64), _c(l, np.float64), _c(o, np.float64)
    lead = m.shape[:-1]
    n_part, D = o.shape[-2], o.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (D,), np.float64)
    _check(_load().oracle_combine_partials(rows, n_part, D, m.ctypes.data, l.ctypes.data, o.ctypes.data,
                                           out.ctypes.data))
    return out


def reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping):
    """In-place slot-mapped append on host pools ([num_blocks][Hkv][bs][D])."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    k_new, v_new = _c(k_new), _c(v_new)
    slots = _c(slot_mapping, np.int64)
    nb, Hkv, bs, D = k_pool.shape
    _check(_load().oracle_reshape_and_cache(k_pool.itemsize, k_new.ctypes.data, v_new.ctypes.data,
                                            k_pool.ctypes.data, v_pool.ctypes.data, slots.ctypes.data,
                                            len(slots), Hkv, D, bs, nb))


def copy_blocks(k_pool, v_pool, pairs):
    """In-place copy-on-write block copies on host pools; pairs is [n][2] (src, dst)."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    pairs = _c(np.asarray(pairs, np.int32).reshape(-1, 2))
    nb, Hkv, bs, D = k_pool.shape
    _check(_load().oracle_copy_blocks(k_pool.itemsize, k_pool.ctypes.data, v_pool.ctypes.data,
                                      pairs.ctypes.data, len(pairs), Hkv, D, bs, nb))
