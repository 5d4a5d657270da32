"""GPU: the allocation-free decode entry point (pa_decode_attention_static).

Callers that cannot allocate device memory -- a plugin whose host framework
owns every allocation, or a serving loop that must not allocate once it is
running -- use this entry point, which keeps its split-sequence scratch in a
static per-GPU buffer inside the library.  These tests call it through the
C ABI twice in a row and compare each result with the regular entry point
(caller-supplied workspace), element by element, within the parity bound of
the other decode tests.  The shapes differ between calls, so a status word or
partial left over in the shared buffer by the previous call would show.
This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import pytest

import synth.workloads as W
from gpu_cases import DecodeCase, check_close, to_numpy, widen

pytestmark = pytest.mark.gpu

CASES = [
    # seed, B, Hq, Hkv, D, bs, dtype, max_len: long sequences so that segments are split across CTAs
    (31, 9, 32, 8, 128, 16, "bf16", 2500),
    (32, 5, 4, 4, 64, 32, "f32", 900),
]


def _run_both(case_args):
    import torch
    import paged_kv_cache_280_gb300 as pa

    seed, B, hq, hkv, d, bs, dtype, max_len = case_args
    w = W.random_case(seed, B, hq, hkv, d, bs, dtype, max_len=max_len, min_len=1)
    c = DecodeCase(w).device()
    c.run()  # regular entry point, caller-owned workspace
    regular = to_numpy(c.dout).copy()
    static_out = torch.full_like(c.dout, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    pa.pa_decode_attention_static(static_out, c.dq, c.dk, c.dv, c.dtables, c.dlens, int(c.lengths.max()), w.scale,
                                  status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return regular, to_numpy(static_out), dtype


def test_static_workspace_matches_regular_entry_point_twice():
    for _ in range(2):  # two calls in a row per shape, shapes alternating
        for args in CASES:
            regular, static, dtype = _run_both(args)
            check_close(static, widen(regular), dtype)


def test_static_workspace_rejects_oversized_scratch():
    import torch
    import paged_kv_cache_280_gb300 as pa

    # 8 query heads per KV head at d 128: two partial slots of 4160 B for each of up to 8 CTAs
    # on every SM (10.1 MB on 152 SMs), more than the 8 MiB static buffer
    B, hq, hkv, d, bs = 4, 64, 8, 128, 16
    assert pa.pa_decode_workspace_bytes(B, hq, hkv, d) > pa.STATIC_WORKSPACE_BYTES
    q = torch.zeros(B, hq, d, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(1, hkv, bs, d, dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_attention_static(out, q, pool, pool, tables, lens, 0, 0.125)
    assert e.value.name == "PA_ERR_WORKSPACE_TOO_SMALL"
