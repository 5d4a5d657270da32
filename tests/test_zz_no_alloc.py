"""GPU: the allocation-free decode entry point (pa_decode_attention_static).

Callers that cannot allocate device memory -- a plugin whose host framework
owns every allocation, or a serving loop that must not allocate once it is
running -- use this entry point, which keeps its split-sequence scratch in a
static per-GPU buffer inside the library.  These tests call it through the
C ABI twice in a row per shape and compare each result with the fp64 oracle
and with the regular entry point (caller-supplied workspace), element by
element, within the parity bound of the other decode tests.  The shapes
differ between calls (split anywhere, fixed partitions, empty sequences, the
64/8-head long-context shape), so a status word or partial left over in the
shared buffer by the previous call would show.
This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

import synth.workloads as W
from gpu_cases import DecodeCase, check_close, to_numpy, widen

pytestmark = pytest.mark.gpu

CASES = [
    # seed, B, Hq, Hkv, D, bs, dtype, min_len, max_len, partition_tokens, empty sequences
    (31, 9, 32, 8, 128, 16, "bf16", 1, 2500, 0, ()),
    (32, 5, 4, 4, 64, 32, "f32", 1, 900, 0, ()),
    (33, 12, 16, 4, 128, 16, "bf16", 0, 3000, 256, (3, 7)),
    # the long-context head shape (64 query / 8 KV heads, d 128) with 2048-token partitions
    (34, 4, 64, 8, 128, 16, "bf16", 32768, 32768, 2048, ()),
]

_cases = {}


def _case(args):
    """Device case, its oracle output and its regular-entry-point output, built once per shape."""
    if args not in _cases:
        seed, B, hq, hkv, d, bs, dtype, lo, hi, pt, empty = args
        w = W.random_case(seed, B, hq, hkv, d, bs, dtype, max_len=hi, min_len=lo)
        lengths = np.asarray(w.lengths, np.int32).copy()
        lengths[list(empty)] = 0
        c = DecodeCase(w, lengths=lengths).device()
        ref = c.oracle(threads=8)
        c.run(partition_tokens=pt)
        _cases[args] = (c, ref, to_numpy(c.dout).copy())
    return _cases[args]


def _static(c, pt):
    import torch
    import paged_kv_cache_280_gb300 as pa

    out = torch.full_like(c.dout, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    pa.pa_decode_attention_static(out, c.dq, c.dk, c.dv, c.dtables, c.dlens, int(c.lengths.max(initial=0)), c.w.scale,
                                  partition_tokens=pt, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return to_numpy(out)


def test_static_workspace_matches_oracle_and_regular_entry_point_twice():
    for _ in range(2):  # two calls in a row per shape, shapes alternating
        for args in CASES:
            c, ref, regular = _case(args)
            got = _static(c, args[9])
            check_close(got, ref, args[6])
            check_close(got, widen(regular), args[6])
            for b in args[10]:
                assert not np.any(widen(got)[b]), "an empty sequence's output is zero"


def test_static_workspace_sizes_by_the_launched_grid():
    """The refusal follows the grid the call launches: per CTA a merge counter and two partial slots of
    G (D + 2) floats, after the 256-byte status head.

    The widest head shape (8 query heads per KV head, d 128) at the most CTAs per SM the kernel can hold
    is checked either way: refused with PA_ERR_WORKSPACE_TOO_SMALL if its grid needs more than the static
    buffer, else run and compared with the oracle."""
    import torch
    import paged_kv_cache_280_gb300 as pa

    B, hq, hkv, d, bs = 4, 64, 8, 128, 16
    w = W.random_case(35, B, hq, hkv, d, bs, "bf16", max_len=4000, min_len=3000)
    c = DecodeCase(w).device()
    ref = c.oracle(threads=8)
    slot_bytes = -(-(hq // hkv) * (d + 2) // 4) * 4 * 4
    try:
        pa.pa_decode_set_ctas_per_sm(8)
        ctas, _, _, _ = pa.pa_decode_launch_info(B, hq, hkv, d, bs, c.max_blocks, pa.PA_BF16)
        need = 256 + -(-4 * ctas // 256) * 256 + 2 * ctas * slot_bytes
        out = torch.full_like(c.dout, float("nan"))
        args = (out, c.dq, c.dk, c.dv, c.dtables, c.dlens, int(c.lengths.max()), w.scale)
        if need > pa.STATIC_WORKSPACE_BYTES:
            with pytest.raises(pa.PAError) as e:
                pa.pa_decode_attention_static(*args)
            assert e.value.name == "PA_ERR_WORKSPACE_TOO_SMALL"
            torch.cuda.synchronize()
            assert torch.isnan(out.float()).all(), "a refused call launches nothing"
        else:
            status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            pa.pa_decode_attention_static(*args, status=status)
            torch.cuda.synchronize()
            assert status.item() == 0
            check_close(to_numpy(out), ref, "bf16")
    finally:
        pa.pa_decode_set_ctas_per_sm(0)
    # at the default CTAs per SM the shape always fits and matches the oracle
    out = torch.full_like(c.dout, float("nan"))
    pa.pa_decode_attention_static(out, c.dq, c.dk, c.dv, c.dtables, c.dlens, int(c.lengths.max()), w.scale)
    torch.cuda.synchronize()
    check_close(to_numpy(out), ref, "bf16")
