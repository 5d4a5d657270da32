"""Python binding of libpa, the paged KV-cache library for one GB300 (sm_103a).

Argument marshalling only: every function here passes tensor data pointers,
sizes and the current CUDA stream to the C ABI declared in ``include/pa.h``
and raises :class:`PAError` on a non-OK status.  All device work happens in
the library's CUDA kernels; there is no fallback path.  The library is built
in-tree by ``__graft_entry__.build()`` (or ``python
paged_kv_cache_280_gb300/_build.py``); importing this package without it raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python paged_kv_cache_280_gb300/_build.py, or __graft_entry__.build())"
    )

_lib = ctypes.CDLL(LIB_PATH)

PA_F32, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
PA_DEV_BAD_BLOCK_ID, PA_DEV_BAD_SLOT, PA_DEV_BAD_SEQ_LEN, PA_DEV_WAIT_TIMEOUT = 1, 2, 4, 8
STATUS_NAMES = {
    0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_OUT_OF_BLOCKS",
    4: "PA_ERR_NO_SUCH_SEQ", 5: "PA_ERR_SEQ_EXISTS", 6: "PA_ERR_REFCOUNT_LIMIT",
    7: "PA_ERR_WORKSPACE_TOO_SMALL", 8: "PA_ERR_BUFFER_TOO_SMALL", 9: "PA_ERR_CUDA", 10: "PA_ERR_INTERNAL",
    11: "PA_ERR_SEQ_SWAPPED",
}


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({_lib.pa_status_str(status).decode()})")


class pa_alloc_stats_t(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
        ("used_blocks", ctypes.c_int32), ("shared_blocks", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
        ("tokens", ctypes.c_int64), ("slots", ctypes.c_int64), ("cow_copies", ctypes.c_int64),
    ]


_i32, _i64, _f32, _vp, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
_pi32, _pi64, _psz = ctypes.POINTER(_i32), ctypes.POINTER(_i64), ctypes.POINTER(_sz)

_SIGS = {
    "pa_reshape_and_cache": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pa_copy_blocks": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pa_decode_workspace_bytes": (_i32, [_i32, _i32, _i32, _i32, _psz]),
    "pa_decode_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                   _f32, _i32, _vp, _sz, _i32, _vp]),
    "pa_decode_attention_static": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                          _i32, _f32, _i32, _i32, _vp, _vp]),
    "pa_decode_launch_info": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _pi32, _pi32, _pi32, _pi32]),
    "pa_decode_kernels_per_call": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _pi32]),
    "pa_decode_plan_bytes": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _psz]),
    "pa_decode_build_plan": (_i32, [_vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz]),
    "pa_decode_attention_planned": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                           _i32, _f32, _i32, _vp, _sz, _i32, _vp, _sz, _vp]),
    "pa_decode_attention_fp8_planned": (_i32, [_vp, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float, _vp, _i32, _vp,
                                               _i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _i32, _vp,
                                               _sz, _vp, _sz, _vp]),
    "pa_seq_create_cached": (_i32, [_vp, _i64, _vp, _i32, _pi32]),
    "pa_seq_cache_prefix": (_i32, [_vp, _i64, _vp, _i32]),
    "pa_prefix_cache_stats": (_i32, [_vp, _pi32, _pi32]),
    "pa_seq_swap_out": (_i32, [_vp, _i64, _vp, _i32, _pi32]),
    "pa_seq_swap_in": (_i32, [_vp, _i64, _vp, _i32, _pi32]),
    "pa_swap_out": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pa_swap_in": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pa_reshape_and_cache_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float,
                                        ctypes.c_float, _vp, _vp]),
    "pa_decode_attention_fp8": (_i32, [_vp, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float, _vp, _i32, _vp, _i32,
                                       _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _i32, _vp, _sz, _vp]),
    "pa_prefill_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                    _i32, _i32, ctypes.c_float, _i32, _vp, _vp]),
    "pa_decode_set_ctas_per_sm": (_i32, [_i32]),
    "pa_debug_set_wait_limit_ns": (_i32, [ctypes.c_uint64]),
    "pa_debug_set_merge_mode": (_i32, [ctypes.c_int32]),
    "pa_debug_set_seg_units": (_i32, [ctypes.c_int32]),
    "pa_debug_set_wave_skew": (_i32, [ctypes.c_int32]),
    "pa_debug_plan_ranges": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "pa_alloc_create": (_i32, [_i32, _i32, _vp, ctypes.POINTER(_vp)]),
    "pa_alloc_destroy": (None, [_vp]),
    "pa_alloc_set_max_refcount": (_i32, [_vp, _i32]),
    "pa_seq_create": (_i32, [_vp, _i64]),
    "pa_seq_append": (_i32, [_vp, _i64, _i32, _vp, _vp, _pi32]),
    "pa_append_batch": (_i32, [_vp, _vp, _i32, _vp, _vp, _pi32]),
    "pa_seq_fork": (_i32, [_vp, _i64, _i64]),
    "pa_seq_free": (_i32, [_vp, _i64]),
    "pa_seq_block_table": (_i32, [_vp, _i64, _vp, _i32, _pi32]),
    "pa_seq_len": (_i32, [_vp, _i64, _pi32]),
    "pa_export_tables": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp]),
    "pa_block_refcount": (_i32, [_vp, _i32]),
    "pa_alloc_stats": (_i32, [_vp, ctypes.POINTER(pa_alloc_stats_t)]),
    "pa_alloc_free_list": (_i32, [_vp, _vp, _i32, _pi32]),
    "pa_status_str": (ctypes.c_char_p, [_i32]),
    "pa_abi_version": (_i32, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def _ok(status: int, where: str) -> None:
    if status != 0:
        raise PAError(status, where)


def abi_version() -> int:
    return int(_lib.pa_abi_version())


# ---------------------------------------------------------------------------
# device entry points (torch tensors on the current CUDA device)
# ---------------------------------------------------------------------------

def _torch():
    import torch

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None):
        return PA_FP8_E4M3
    raise PAError(2, f"dtype {t.dtype}")


def _dev_ptr(t, name: str) -> int:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _acc_ptr(t, name: str) -> int:
    """Pointer to a tensor the GPU can address: CUDA memory or pinned host memory."""
    if t is None:
        return None
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pa_reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping, status=None, stream=None):
    """k_new/v_new [N][Hkv][D]; pools [num_blocks][Hkv][bs][D]; slot_mapping int64 [N]."""
    nb, hkv, bs, d = k_pool.shape
    n = slot_mapping.shape[0]
    _ok(_lib.pa_reshape_and_cache(_dev_ptr(k_new, "k_new"), _dev_ptr(v_new, "v_new"), _dev_ptr(k_pool, "k_pool"),
                                  _dev_ptr(v_pool, "v_pool"), _dev_ptr(slot_mapping, "slot_mapping"), n, hkv, d, bs,
                                  nb, _dtype_code(k_pool), _dev_ptr(status, "status"), _stream(stream)),
        "pa_reshape_and_cache")


def pa_copy_blocks(k_pool, v_pool, src_dst_pairs, status=None, stream=None):
    """src_dst_pairs int32 [n][2] on the device."""
    nb, hkv, bs, d = k_pool.shape
    n = src_dst_pairs.shape[0]
    _ok(_lib.pa_copy_blocks(_dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"),
                            _dev_ptr(src_dst_pairs, "src_dst_pairs"), n, hkv, d, bs, nb, _dtype_code(k_pool),
                            _dev_ptr(status, "status"), _stream(stream)),
        "pa_copy_blocks")


def pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim) -> int:
    out = _sz(0)
    _ok(_lib.pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, ctypes.byref(out)),
        "pa_decode_workspace_bytes")
    return int(out.value)


def pa_decode_attention(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len, scale, workspace,
                        partition_tokens=0, stream=None, plan=None):
    """out/q [B][Hq][D]; pools [num_blocks][Hkv][bs][D]; block_tables int32 [B][max_blocks]; seq_lens int32 [B];
    workspace: a zero-initialised uint8 CUDA tensor of pa_decode_workspace_bytes bytes.  plan: optional device copy
    (int32 CUDA tensor) of a pa_decode_build_plan result for this call."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_pool.shape
    args = [_dev_ptr(out, "out"), _dev_ptr(q, "q"), _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"),
            _dev_ptr(block_tables, "block_tables"), block_tables.shape[1], _dev_ptr(seq_lens, "seq_lens"),
            int(max_seq_len), b, hq, hkv, d, bs, nb, float(scale), int(partition_tokens),
            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(), _dtype_code(q)]
    if plan is None:
        _ok(_lib.pa_decode_attention(*args, _stream(stream)), "pa_decode_attention")
    else:
        _ok(_lib.pa_decode_attention_planned(*args, _dev_ptr(plan, "plan"), plan.numel() * plan.element_size(),
                                             _stream(stream)), "pa_decode_attention_planned")


def pa_decode_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, max_seq_len,
                         partition_tokens, dtype):
    n = _sz(0)
    _ok(_lib.pa_decode_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                  int(max_seq_len), int(partition_tokens), dtype, ctypes.byref(n)),
        "pa_decode_plan_bytes")
    return int(n.value)


def pa_decode_build_plan(block_tables, seq_lens, max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size,
                         partition_tokens, dtype, out=None):
    """The decode plan (int32 numpy array) from host copies of the block tables ([B][max_blocks] int32) and
    lengths ([B] int32).  ``out``: an int32 numpy array (e.g. a view of a pinned staging buffer) to write into,
    of pa_decode_plan_bytes bytes at least (shorter raises PAError: PA_ERR_WORKSPACE_TOO_SMALL); without it the
    plan's size is asked for first."""
    import numpy as np

    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    b, mb = tables.shape
    if out is None:
        n = pa_decode_plan_bytes(b, num_q_heads, num_kv_heads, head_dim, block_size, mb, max_seq_len,
                                 partition_tokens, dtype)
        out = np.empty(n // 4, dtype=np.int32)
    if out.dtype != np.int32 or not out.flags["C_CONTIGUOUS"]:
        raise ValueError("pa_decode_build_plan: out must be a contiguous int32 array")
    _ok(_lib.pa_decode_build_plan(tables.ctypes.data, mb, lens.ctypes.data, int(max_seq_len), b, num_q_heads,
                                  num_kv_heads, head_dim, block_size, int(partition_tokens), dtype, out.ctypes.data,
                                  out.nbytes), "pa_decode_build_plan")
    return out


STATIC_WORKSPACE_BYTES = 8 << 20


def pa_decode_attention_static(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len, scale,
                               partition_tokens=0, status=None, stream=None):
    """pa_decode_attention without a workspace argument, for callers that cannot allocate device memory.

    The library's own per-GPU static scratch (STATIC_WORKSPACE_BYTES) is used; calls that overlap on the GPU
    race on it.  ``status``: optional int32 CUDA tensor that receives the device status word."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_pool.shape
    _ok(_lib.pa_decode_attention_static(_dev_ptr(out, "out"), _dev_ptr(q, "q"), _dev_ptr(k_pool, "k_pool"),
                                        _dev_ptr(v_pool, "v_pool"), _dev_ptr(block_tables, "block_tables"),
                                        block_tables.shape[1], _dev_ptr(seq_lens, "seq_lens"), int(max_seq_len), b,
                                        hq, hkv, d, bs, nb, float(scale), int(partition_tokens), _dtype_code(q),
                                        _dev_ptr(status, "status"), _stream(stream)),
        "pa_decode_attention_static")


def pa_decode_launch_info(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype,
                          partition_tokens=0):
    """(ctas, stages, smem_bytes, uses_mma) of a decode call with these shapes on the current device."""
    vals = [_i32(0) for _ in range(4)]
    _ok(_lib.pa_decode_launch_info(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                   int(partition_tokens), dtype, *[ctypes.byref(v) for v in vals]),
        "pa_decode_launch_info")
    return tuple(int(v.value) for v in vals)


def pa_decode_kernels_per_call(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                               partition_tokens, dtype):
    """1 if a decode call with these shapes merges split segments in the decode kernel, 2 if a merge kernel follows."""
    v = _i32(0)
    _ok(_lib.pa_decode_kernels_per_call(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                        int(partition_tokens), dtype, ctypes.byref(v)), "pa_decode_kernels_per_call")
    return int(v.value)


def pa_reshape_and_cache_fp8(k_new, v_new, k_pool, v_pool, slot_mapping, k_scale, v_scale, status=None,
                             stream=None):
    """Slot-mapped append into FP8 pools (uint8 E4M3 codes [num_blocks][Hkv][bs][128]) of bf16/fp32 K/V."""
    nb, hkv, bs, d = k_pool.shape
    n = slot_mapping.shape[0]
    _ok(_lib.pa_reshape_and_cache_fp8(_dev_ptr(k_new, "k_new"), _dev_ptr(v_new, "v_new"), _dev_ptr(k_pool, "k_pool"),
                                      _dev_ptr(v_pool, "v_pool"), _dev_ptr(slot_mapping, "slot_mapping"), n, hkv, d,
                                      bs, nb, _dtype_code(k_new), float(k_scale), float(v_scale),
                                      _dev_ptr(status, "status"), _stream(stream)),
        "pa_reshape_and_cache_fp8")


def pa_decode_attention_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, max_seq_len, scale,
                            workspace, partition_tokens=0, stream=None, plan=None):
    """Decode over FP8 pools (uint8 E4M3 codes) with bf16 q/out; K^ = code value * k_scale, V^ likewise.
    plan: as for pa_decode_attention (built with dtype PA_FP8_E4M3)."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_pool.shape
    args = [_dev_ptr(out, "out"), _dev_ptr(q, "q"), _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"),
            float(k_scale), float(v_scale), _dev_ptr(block_tables, "block_tables"), block_tables.shape[1],
            _dev_ptr(seq_lens, "seq_lens"), int(max_seq_len), b, hq, hkv, d, bs, nb, float(scale),
            int(partition_tokens), _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()]
    if plan is None:
        _ok(_lib.pa_decode_attention_fp8(*args, _stream(stream)), "pa_decode_attention_fp8")
    else:
        _ok(_lib.pa_decode_attention_fp8_planned(*args, _dev_ptr(plan, "plan"), plan.numel() * plan.element_size(),
                                                 _stream(stream)), "pa_decode_attention_fp8_planned")


def pa_swap_out(k_pool, v_pool, blocks, k_store, v_store, status=None, stream=None):
    """store[i] = pool[blocks[i]] (whole blocks, K and V).  Stores [n][Hkv][bs][D] and blocks int32 [n] may be
    CUDA tensors or pinned host tensors."""
    nb, hkv, bs, d = k_pool.shape
    _ok(_lib.pa_swap_out(_dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"), _acc_ptr(blocks, "blocks"),
                         blocks.shape[0], _acc_ptr(k_store, "k_store"), _acc_ptr(v_store, "v_store"), hkv, d, bs, nb,
                         _dtype_code(k_pool), _dev_ptr(status, "status"), _stream(stream)),
        "pa_swap_out")


def pa_swap_in(k_store, v_store, blocks, k_pool, v_pool, status=None, stream=None):
    """pool[blocks[i]] = store[i] (whole blocks, K and V); the inverse of pa_swap_out."""
    nb, hkv, bs, d = k_pool.shape
    _ok(_lib.pa_swap_in(_acc_ptr(k_store, "k_store"), _acc_ptr(v_store, "v_store"), _acc_ptr(blocks, "blocks"),
                        blocks.shape[0], _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"), hkv, d, bs, nb,
                        _dtype_code(k_pool), _dev_ptr(status, "status"), _stream(stream)),
        "pa_swap_in")


def pa_prefill_attention(out, q, k_pool, v_pool, block_tables, seq_lens, cu_q_lens, max_q_len, scale, status=None,
                         stream=None):
    """Paged prefill (chunked causal) attention, bf16.  out/q [T][Hq][D]; pools [num_blocks][Hkv][bs][D];
    block_tables int32 [B][max_blocks]; seq_lens int32 [B] (context incl. the chunk); cu_q_lens int32 [B+1]."""
    t, hq, d = q.shape
    nb, hkv, bs, _ = k_pool.shape
    b = seq_lens.shape[0]
    _ok(_lib.pa_prefill_attention(_dev_ptr(out, "out"), _dev_ptr(q, "q"), _dev_ptr(k_pool, "k_pool"),
                                  _dev_ptr(v_pool, "v_pool"), _dev_ptr(block_tables, "block_tables"),
                                  block_tables.shape[1], _dev_ptr(seq_lens, "seq_lens"), _dev_ptr(cu_q_lens, "cu_q_lens"),
                                  b, t, int(max_q_len), hq, hkv, d, bs, nb, float(scale), _dtype_code(q),
                                  _dev_ptr(status, "status"), _stream(stream)),
        "pa_prefill_attention")


def pa_decode_set_ctas_per_sm(ctas: int) -> None:
    _ok(_lib.pa_decode_set_ctas_per_sm(int(ctas)), "pa_decode_set_ctas_per_sm")


def pa_debug_set_wait_limit_ns(ns: int) -> None:
    """Testing aid: time limit of the decode consumer's waits (0 restores the 2 s default)."""
    _ok(_lib.pa_debug_set_wait_limit_ns(int(ns)), "pa_debug_set_wait_limit_ns")


MERGE_AUTO, MERGE_IN_KERNEL, MERGE_KERNEL = 0, 1, 2


def pa_debug_set_merge_mode(mode: int) -> None:
    """Testing aid: where decode calls merge split segments (MERGE_AUTO, MERGE_IN_KERNEL or MERGE_KERNEL)."""
    _ok(_lib.pa_debug_set_merge_mode(int(mode)), "pa_debug_set_merge_mode")


def pa_debug_set_seg_units(units: int) -> None:
    """Tuning aid: a segment's weight in the balance of the decode's CTA ranges (a tile weighs 4); 0 restores
    each compute path's own."""
    _ok(_lib.pa_debug_set_seg_units(int(units)), "pa_debug_set_seg_units")


def pa_debug_plan_ranges(block_counts, num_kv_heads, partition_tiles, seg_units, num_ctas, wave_ctas, wave_skew,
                         owners=True):
    """Testing aid (no GPU): (range starts [W + 1] int64, owners [T] int32 or None) of a decode launch's CTA
    ranges, W the working CTAs, from per-sequence block counts."""
    import numpy as np

    counts = np.ascontiguousarray(block_counts, dtype=np.int32)
    starts = np.zeros(int(num_ctas) + 1, np.int64)
    total = int(counts.sum()) * int(num_kv_heads)
    own = np.zeros(max(total, 1), np.int32) if owners else None
    working = ctypes.c_int32(0)
    _ok(_lib.pa_debug_plan_ranges(counts.ctypes.data, len(counts), int(num_kv_heads), int(partition_tiles),
                                  int(seg_units), int(num_ctas), int(wave_ctas), int(wave_skew), starts.ctypes.data,
                                  own.ctypes.data if owners else None, own.size if owners else 0,
                                  ctypes.byref(working)), "pa_debug_plan_ranges")
    return starts[: working.value + 1], (own[:total] if owners else None)


def pa_debug_set_wave_skew(skew: int) -> None:
    """Tuning aid: the skew of the decode's CTA shares by dispatch wave (0: equal shares); -1 restores each
    compute path's own."""
    _ok(_lib.pa_debug_set_wave_skew(int(skew)), "pa_debug_set_wave_skew")


# ---------------------------------------------------------------------------
# host allocator
# ---------------------------------------------------------------------------

def _np():
    import numpy as np

    return np


def _int64_array(seq_ids):
    np = _np()
    if isinstance(seq_ids, np.ndarray) and seq_ids.dtype == np.int64 and seq_ids.flags["C_CONTIGUOUS"]:
        return seq_ids
    return np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))


def _checked_out(a, dtype, n: int, cols: int):
    """A caller-provided output array: C-contiguous, of dtype, with room for n rows of ``cols``."""
    np = _np()
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags["C_CONTIGUOUS"] or a.size < max(1, n) * cols:
        raise ValueError(f"output array must be C-contiguous {np.dtype(dtype).name} with room for {n} x {cols}")
    return a.reshape(-1, cols) if cols > 1 else a.reshape(-1)


class Allocator:
    """Host block allocator (pa_alloc_*): on-demand blocks, block tables, refcounts, copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None, max_refcount: int = 0):
        np = _np()
        self._h = _vp()
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
            if order.shape != (num_blocks,):
                raise ValueError("free_order must hold num_blocks ids")
        _ok(_lib.pa_alloc_create(num_blocks, block_size, None if order is None else order.ctypes.data,
                                 ctypes.byref(self._h)), "pa_alloc_create")
        self.num_blocks = num_blocks
        self.block_size = block_size
        if max_refcount:
            _ok(_lib.pa_alloc_set_max_refcount(self._h, max_refcount), "pa_alloc_set_max_refcount")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.pa_alloc_destroy(h)
            self._h = None

    def create(self, seq_id: int) -> None:
        _ok(_lib.pa_seq_create(self._h, seq_id), "pa_seq_create")

    def append(self, seq_id: int, n_tokens: int):
        """Returns (slots int64 [n], cow_pairs int32 [k][2])."""
        np = _np()
        slots = np.empty(max(1, n_tokens), np.int64)
        pairs = np.empty((max(1, n_tokens), 2), np.int32)
        n_cow = _i32(0)
        _ok(_lib.pa_seq_append(self._h, seq_id, n_tokens, slots.ctypes.data, pairs.ctypes.data, ctypes.byref(n_cow)),
            "pa_seq_append")
        return slots[:n_tokens], pairs[: n_cow.value]

    def append_batch(self, seq_ids, slots_out=None, pairs_out=None):
        """One token per id, in order.  Returns (slots int64 [n], cow_pairs int32 [k][2]).

        ``slots_out`` (int64, >= n entries) and ``pairs_out`` (int32 [>= n][2]),
        when given, receive the results in place (e.g. pinned staging buffers).
        """
        np = _np()
        ids = _int64_array(seq_ids)
        n = len(ids)
        slots = np.empty(max(1, n), np.int64) if slots_out is None else _checked_out(slots_out, np.int64, n, 1)
        pairs = np.empty((max(1, n), 2), np.int32) if pairs_out is None else _checked_out(pairs_out, np.int32, n, 2)
        n_cow = _i32(0)
        _ok(_lib.pa_append_batch(self._h, ids.ctypes.data, n, slots.ctypes.data, pairs.ctypes.data,
                                 ctypes.byref(n_cow)), "pa_append_batch")
        return slots[:n], pairs[: n_cow.value]

    def fork(self, parent: int, child: int) -> None:
        _ok(_lib.pa_seq_fork(self._h, parent, child), "pa_seq_fork")

    def free_seq(self, seq_id: int) -> None:
        _ok(_lib.pa_seq_free(self._h, seq_id), "pa_seq_free")

    def create_cached(self, seq_id: int, tokens) -> int:
        """Create a sequence starting with the longest cached run of full blocks of ``tokens``; returns the
        tokens covered (the new sequence's length)."""
        np = _np()
        tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = _i32(0)
        _ok(_lib.pa_seq_create_cached(self._h, seq_id, tk.ctypes.data if tk.size else None, tk.size, ctypes.byref(n)),
            "pa_seq_create_cached")
        return int(n.value)

    def cache_prefix(self, seq_id: int, tokens) -> None:
        """Register the full blocks of the sequence's first len(tokens) tokens in the prefix cache."""
        np = _np()
        tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        _ok(_lib.pa_seq_cache_prefix(self._h, seq_id, tk.ctypes.data if tk.size else None, tk.size),
            "pa_seq_cache_prefix")

    def prefix_cache_stats(self) -> dict:
        c, e = _i32(0), _i32(0)
        _ok(_lib.pa_prefix_cache_stats(self._h, ctypes.byref(c), ctypes.byref(e)), "pa_prefix_cache_stats")
        return {"cached_blocks": int(c.value), "evictable_blocks": int(e.value)}

    def swap_out(self, seq_id: int):
        """Release the sequence's blocks for a swap-out; returns their ids (int32, logical order) to copy out."""
        np = _np()
        n = _i32(0)
        cap = self.length(seq_id) // self.block_size + 1
        out = np.empty(max(1, cap), np.int32)
        _ok(_lib.pa_seq_swap_out(self._h, seq_id, out.ctypes.data, cap, ctypes.byref(n)), "pa_seq_swap_out")
        return out[: n.value]

    def swap_in(self, seq_id: int):
        """Give a swapped-out sequence fresh blocks; returns their ids (int32, logical order) to copy back into."""
        np = _np()
        n = _i32(0)
        cap = self.length(seq_id) // self.block_size + 1
        out = np.empty(max(1, cap), np.int32)
        _ok(_lib.pa_seq_swap_in(self._h, seq_id, out.ctypes.data, cap, ctypes.byref(n)), "pa_seq_swap_in")
        return out[: n.value]

    def length(self, seq_id: int) -> int:
        n = _i32(0)
        _ok(_lib.pa_seq_len(self._h, seq_id, ctypes.byref(n)), "pa_seq_len")
        return int(n.value)

    def table(self, seq_id: int):
        np = _np()
        cap = self.length(seq_id) // self.block_size + 1
        out = np.empty(max(1, cap), np.int32)
        n = _i32(0)
        _ok(_lib.pa_seq_block_table(self._h, seq_id, out.ctypes.data, cap, ctypes.byref(n)), "pa_seq_block_table")
        return out[: n.value].tolist()

    def export_tables(self, seq_ids, max_blocks_per_seq: int, tables_out=None, lens_out=None):
        """(tables int32 [n][max_blocks_per_seq], lens int32 [n]) in the decode kernel's layout.

        ``tables_out`` / ``lens_out``, when given (C-contiguous int32 arrays of
        exactly those shapes), are filled in place.
        """
        np = _np()
        ids = _int64_array(seq_ids)
        n = len(ids)
        tables = np.empty((n, max_blocks_per_seq), np.int32) if tables_out is None else tables_out
        lens = np.empty(n, np.int32) if lens_out is None else lens_out
        if tables_out is not None or lens_out is not None:
            for a, shape in ((tables, (n, max_blocks_per_seq)), (lens, (n,))):
                if a.dtype != np.int32 or a.shape != shape or not a.flags["C_CONTIGUOUS"]:
                    raise ValueError(f"output arrays must be C-contiguous int32 of shape {shape}")
        _ok(_lib.pa_export_tables(self._h, ids.ctypes.data, len(ids), max_blocks_per_seq, tables.ctypes.data,
                                  lens.ctypes.data), "pa_export_tables")
        return tables, lens

    def refcount(self, block: int) -> int:
        return int(_lib.pa_block_refcount(self._h, block))

    def free_list(self):
        np = _np()
        out = np.empty(max(1, self.num_blocks), np.int32)
        n = _i32(0)
        _ok(_lib.pa_alloc_free_list(self._h, out.ctypes.data, self.num_blocks, ctypes.byref(n)), "pa_alloc_free_list")
        return out[: n.value].tolist()

    def stats(self) -> dict:
        s = pa_alloc_stats_t()
        _ok(_lib.pa_alloc_stats(self._h, ctypes.byref(s)), "pa_alloc_stats")
        return {name: int(getattr(s, name)) for name, _ in s._fields_}
