"""GPU: decode calls with a host-built plan (pa_decode_build_plan) give the same bits as the calls
without one, on every compute path, with and without fixed partitions, in both merge modes; a
plan for other shapes is ignored; the plan's own words follow from the lengths and tables alone."""
import numpy as np
import pytest

import oracle
import synth.workloads as W
from gpu_cases import DecodeCase, check_close, status_word, to_numpy, to_torch
from test_gpu_fp8 import _fp8_case

pytestmark = pytest.mark.gpu


def _dtype_code(pa, dtype):
    return {"bf16": pa.PA_BF16, "f32": pa.PA_F32, "fp8": pa.PA_FP8_E4M3}[dtype]


def _decode(c, pa, dtype, pt, plan=None, max_len=None):
    import torch

    ml = int(c.lengths.max(initial=0)) if max_len is None else max_len
    n = pa.pa_decode_workspace_bytes(len(c.lengths), c.w.num_q_heads, c.w.num_kv_heads, c.w.head_dim)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    dplan = None if plan is None else torch.from_numpy(plan).cuda()
    if dtype == "fp8":
        dq, dt, dl = to_torch(c.q), to_torch(c.tables), to_torch(c.lengths)
        dk, dv = torch.from_numpy(c.kq).cuda(), torch.from_numpy(c.vq).cuda()
        out = torch.full_like(dq, float("nan"))
        pa.pa_decode_attention_fp8(out, dq, dk, dv, *c.scales, dt, dl, ml, c.w.scale, ws, partition_tokens=pt,
                                   plan=dplan)
    else:
        c.device()
        out = torch.full_like(c.dq, float("nan"))
        pa.pa_decode_attention(out, c.dq, c.dk, c.dv, c.dtables, c.dlens, ml, c.w.scale, ws, partition_tokens=pt,
                               plan=dplan)
    torch.cuda.synchronize()
    assert status_word(ws) == 0
    return to_numpy(out)


CASES = [  # dtype, hq, hkv, d, bs, partition tokens
    ("bf16", 32, 8, 128, 16, 0),     # tensor cores
    ("bf16", 32, 8, 128, 16, 256),   # fixed partitions
    ("bf16", 8, 8, 128, 16, 0),      # CUDA cores, G = 1
    ("bf16", 16, 2, 64, 32, 0),
    ("f32", 8, 2, 128, 16, 0),
    ("fp8", 32, 8, 128, 16, 0),
    ("fp8", 64, 8, 128, 16, 512),
]


@pytest.mark.parametrize("merge", [0, 1, 2])
@pytest.mark.parametrize("dtype,hq,hkv,d,bs,pt", CASES)
def test_planned_decode_matches_unplanned_bit_for_bit(dtype, hq, hkv, d, bs, pt, merge):
    import paged_kv_cache_280_gb300 as pa

    lens = np.asarray([700, 0, 1, 33, 1500, 16, 17, 260, 0, 999, 64, 5], np.int32)
    if dtype == "fp8":
        c = _fp8_case(71 + hq, hq, hkv, bs, lens=lens, max_len=1500)
    else:
        w = W.random_case(71 + hq + d, len(lens), hq, hkv, d, bs, dtype, max_len=1500, min_len=1)
        c = DecodeCase(w, lengths=lens)
    ml = int(lens.max())
    try:
        pa.pa_debug_set_merge_mode(merge)
        pa.pa_decode_set_ctas_per_sm(8)
        plan = pa.pa_decode_build_plan(c.tables, c.lengths, ml, hq, hkv, d, bs, pt, _dtype_code(pa, dtype))
        base = _decode(c, pa, dtype, pt)
        got = _decode(c, pa, dtype, pt, plan=plan)
        assert np.array_equal(base.view(np.uint8), got.view(np.uint8))
        # a plan built for another length bound names another launch: ignored, same bits
        other = pa.pa_decode_build_plan(c.tables, c.lengths, ml + 16 * bs, hq, hkv, d, bs, pt, _dtype_code(pa, dtype))
        assert np.array_equal(base.view(np.uint8), _decode(c, pa, dtype, pt, plan=other).view(np.uint8))
    finally:
        pa.pa_debug_set_merge_mode(0)
        pa.pa_decode_set_ctas_per_sm(0)
    if dtype != "fp8":
        check_close(got, c.oracle(), dtype)


def test_plan_words_follow_the_batch():
    """Header, clamped lengths and block prefix sums as the scan would make them; every record's range ends
    tile the batch in order; a record's first chunk holds the table entries of its range's first tiles."""
    import paged_kv_cache_280_gb300 as pa

    lens = np.asarray([40, 0, 2000, 3, 17], np.int32)
    B, hq, hkv, d, bs = len(lens), 16, 4, 128, 16
    w = W.random_case(5, B, hq, hkv, d, bs, "bf16", max_len=2000, min_len=1)
    c = DecodeCase(w, lengths=lens)
    plan = pa.pa_decode_build_plan(c.tables, lens, 1000, hq, hkv, d, bs, 0, pa.PA_BF16)  # clamps 2000 to 1000
    assert plan[0] == 0x4C504150 and plan[1] == B and plan[3] == hkv and plan[7] == 1000
    grid = int(plan[2])
    assert plan.nbytes == pa.pa_decode_plan_bytes(B, hq, hkv, d, bs, c.tables.shape[1], 1000, 0, pa.PA_BF16)
    arr = plan[16:]
    clamped = np.minimum(lens, 1000)
    nblk = (clamped + bs - 1) // bs
    assert np.array_equal(arr[: B + 1], np.concatenate([[0], np.cumsum(nblk)]))
    assert np.array_equal(arr[2 * B + 2: 3 * B + 2], clamped)
    recs = plan[16 + 3 * B + 2:].reshape(grid, 40)
    T = hkv * int(nblk.sum())
    t0, t1 = recs[:, 0], recs[:, 1]
    work = t1 > t0
    assert t0[work][0] == 0 and t1[work][-1] == T
    assert np.array_equal(t0[work][1:], t1[work][:-1])  # consecutive, no gap, no overlap
    # the first chunk of each working range: entries of its first tiles (tiles are sequence-major, then head)
    pref = np.concatenate([[0], np.cumsum(nblk)])
    for r in recs[work]:
        t = int(r[0])
        b = int(np.searchsorted(hkv * pref, t, side="right") - 1)
        while hkv * pref[b + 1] <= t:
            b += 1
        local = t - hkv * pref[b]
        j0 = local % nblk[b]
        n = min(32, nblk[b] - j0, int(r[1]) - t)
        assert np.array_equal(r[8: 8 + n], c.tables[b, j0: j0 + n])


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_matching_plan_is_read(dtype):
    """A plan whose header matches is what the kernel follows: pointing every record's first chunk at
    another (valid) pool block changes the output, and the same plan with a mismatched header does not."""
    import paged_kv_cache_280_gb300 as pa

    lens = np.asarray([700, 33, 1500, 260, 999, 64], np.int32)
    hq, hkv, d, bs = 32, 8, 128, 16
    if dtype == "fp8":
        c = _fp8_case(91, hq, hkv, bs, lens=lens, max_len=1500)
    else:
        c = DecodeCase(W.random_case(91, len(lens), hq, hkv, d, bs, dtype, max_len=1500, min_len=1), lengths=lens)
    ml = int(lens.max())
    plan = pa.pa_decode_build_plan(c.tables, c.lengths, ml, hq, hkv, d, bs, 0, _dtype_code(pa, dtype))
    B, grid = len(lens), int(plan[2])
    recs = plan[16 + 3 * B + 2:].reshape(grid, 40)
    other = int(c.tables[0, 0])  # a valid block of the pool: every read stays in bounds
    bent = plan.copy()
    brecs = bent[16 + 3 * B + 2:].reshape(grid, 40)
    brecs[:, 8:] = np.where(recs[:, 8:] != 0, other, 0)
    assert (brecs[:, 8:] != recs[:, 8:]).any()
    base = _decode(c, pa, dtype, 0)
    assert not np.array_equal(base.view(np.uint8), _decode(c, pa, dtype, 0, plan=bent).view(np.uint8))
    bent[1] += 1  # another batch size in the header: the plan is not used
    assert np.array_equal(base.view(np.uint8), _decode(c, pa, dtype, 0, plan=bent).view(np.uint8))


@pytest.mark.parametrize("units", [1, 24, 4096])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_segment_weight_moves_ranges_not_results(dtype, units):
    """Another segment weight gives other CTA ranges (so other splits and merges), outputs within the
    tolerance of the oracle's, and a plan built under it matches the unplanned call bit for bit."""
    import paged_kv_cache_280_gb300 as pa

    lens = np.asarray([700, 0, 1, 33, 1500, 16, 17, 260, 0, 999, 64, 5], np.int32)
    hq, hkv, d, bs = 32, 8, 128, 16
    if dtype == "fp8":
        c = _fp8_case(73, hq, hkv, bs, lens=lens, max_len=1500)
    else:
        c = DecodeCase(W.random_case(73, len(lens), hq, hkv, d, bs, dtype, max_len=1500, min_len=1), lengths=lens)
    ml = int(lens.max())
    try:
        pa.pa_debug_set_seg_units(units)
        pa.pa_decode_set_ctas_per_sm(8)
        plan = pa.pa_decode_build_plan(c.tables, c.lengths, ml, hq, hkv, d, bs, 0, _dtype_code(pa, dtype))
        assert plan[5] == units
        base = _decode(c, pa, dtype, 0)
        got = _decode(c, pa, dtype, 0, plan=plan)
    finally:
        pa.pa_debug_set_seg_units(0)
        pa.pa_decode_set_ctas_per_sm(0)
    assert np.array_equal(base.view(np.uint8), got.view(np.uint8))
    if dtype == "fp8":
        ref = oracle.decode_attention_fp8(c.q, c.kq, c.vq, *c.scales, c.ref_tables, c.lengths, c.w.scale, threads=8)
        check_close(got, ref, "bf16")
    else:
        check_close(got, c.oracle(), dtype)


@pytest.mark.parametrize("skew", [0, 3, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_wave_shares_move_ranges_not_results(dtype, skew):
    """CTA shares skewed by dispatch wave: outputs within the oracle's tolerance, and a plan built under the
    same skew matches the unplanned call bit for bit."""
    import paged_kv_cache_280_gb300 as pa

    lens = np.asarray([700, 0, 1, 33, 1500, 16, 17, 260, 0, 999, 64, 5, 1200, 800], np.int32)
    hq, hkv, d, bs = 32, 8, 128, 16
    if dtype == "fp8":
        c = _fp8_case(75, hq, hkv, bs, lens=lens, max_len=1500)
    else:
        c = DecodeCase(W.random_case(75, len(lens), hq, hkv, d, bs, dtype, max_len=1500, min_len=1), lengths=lens)
    ml = int(lens.max())
    try:
        pa.pa_debug_set_wave_skew(skew)
        plan = pa.pa_decode_build_plan(c.tables, c.lengths, ml, hq, hkv, d, bs, 0, _dtype_code(pa, dtype))
        assert plan[11] == skew
        base = _decode(c, pa, dtype, 0)
        got = _decode(c, pa, dtype, 0, plan=plan)
    finally:
        pa.pa_debug_set_wave_skew(-1)
    assert np.array_equal(base.view(np.uint8), got.view(np.uint8))
    if dtype == "fp8":
        ref = oracle.decode_attention_fp8(c.q, c.kq, c.vq, *c.scales, c.ref_tables, c.lengths, c.w.scale, threads=8)
        check_close(got, ref, "bf16")
    else:
        check_close(got, c.oracle(), dtype)
