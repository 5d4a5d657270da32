"""GPU: paged decode attention against the fp64 oracle, element by element.

Small ragged cases cover every compiled variant (fp32/bf16, head_dim 64/128,
block 16/32, CUDA-core and tensor-core paths, 1..8 query heads per KV head),
both split modes, several grid sizes, and the edge cases (empty sequences,
one token, exact block multiples, a bad table entry, bad lengths).
"""
import math

import numpy as np
import pytest

import synth.workloads as W
from gpu_cases import DecodeCase, check_close, poison_unused_slots, status_word, to_numpy, to_torch

pytestmark = pytest.mark.gpu

VARIANTS = [
    # dtype, Hq, Hkv, D, bs   (bf16 with Hq/Hkv >= 4 takes the tensor-core path)
    ("f32", 4, 4, 64, 16),
    ("f32", 8, 2, 128, 32),
    ("f32", 16, 2, 64, 32),
    ("f32", 3, 1, 128, 16),
    ("bf16", 4, 4, 128, 16),
    ("bf16", 6, 2, 64, 16),
    ("bf16", 4, 1, 128, 16),
    ("bf16", 8, 1, 128, 32),
    ("bf16", 16, 2, 64, 32),
    ("bf16", 32, 8, 128, 16),
    ("bf16", 5, 1, 64, 16),
    ("bf16", 2, 2, 64, 32),
]


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", VARIANTS)
def test_variants_ragged(dtype, hq, hkv, d, bs):
    w = W.random_case(100 + hq + d + bs, 13, hq, hkv, d, bs, dtype, max_len=300)
    lens = w.lengths.copy()
    lens[:6] = [0, 1, bs - 1, bs, bs + 1, 2 * bs]  # edge lengths
    c = DecodeCase(w, lengths=lens).device()
    ws = c.run()
    ref = c.oracle()
    check_close(to_numpy(c.dout), ref, dtype)
    assert status_word(ws) == 0
    assert np.array_equal(to_numpy(c.dout)[0], np.zeros_like(to_numpy(c.dout)[0]))  # empty sequence -> 0


def test_tiny_fp32_workload():
    """4 sequences {5, 17, 33, 48}, MHA 4 heads, d 64, fp32, 32-block permuted pool: |err| <= 1e-5."""
    c = DecodeCase(W.tiny_fp32()).device()
    ws = c.run()
    err = check_close(to_numpy(c.dout), c.oracle(), "f32")
    assert err <= 1e-5 and status_word(ws) == 0


@pytest.mark.parametrize("merge", [1, 2])  # in the decode kernel; by the merge kernel
@pytest.mark.parametrize("partition_tokens", [0, 16, 32, 64, 2048])
@pytest.mark.parametrize("ctas", [1, 2, 5, 8])
def test_split_modes_and_grid_sizes(partition_tokens, ctas, merge):
    import paged_kv_cache_280_gb300 as pa

    w = W.random_case(7, 9, 16, 2, 128, 16, "bf16", max_len=2500, min_len=1)
    c = DecodeCase(w).device()
    ref = c.oracle()
    try:
        pa.pa_decode_set_ctas_per_sm(ctas)
        pa.pa_debug_set_merge_mode(merge)
        ws = c.run(partition_tokens=partition_tokens)
        first = to_numpy(c.dout).copy()
        c.dout.fill_(float("nan"))
        c.run(ws=ws, partition_tokens=partition_tokens)  # workspace reused
        assert np.array_equal(first, to_numpy(c.dout))  # deterministic merge order, every row rewritten
    finally:
        pa.pa_decode_set_ctas_per_sm(0)
        pa.pa_debug_set_merge_mode(0)
    check_close(first, ref, "bf16")
    # every merge counter (one int32 per CTA after the 256-byte status head) is back at zero
    import torch

    ctas = 8 * torch.cuda.get_device_properties(0).multi_processor_count
    assert not to_numpy(ws[256:256 + 4 * ctas].view(torch.int32)).any()


def test_kernels_per_call_follows_the_merge_mode():
    """Fixed partitions and fp32 pools merge with the second kernel; the testing knob forces either mode
    where both are built; many segments per CTA merge in the decode kernel."""
    import paged_kv_cache_280_gb300 as pa

    assert pa.pa_decode_kernels_per_call(4, 64, 8, 128, 16, 8192, 2048, pa.PA_BF16) == 2
    assert pa.pa_decode_kernels_per_call(64, 16, 4, 128, 16, 64, 0, pa.PA_F32) == 2
    assert pa.pa_decode_kernels_per_call(256, 32, 32, 128, 16, 64, 0, pa.PA_BF16) == 1  # 8192 segments
    # FP8 pools: the merge kernel (the build with three consumer warps per CTA)
    assert pa.pa_decode_kernels_per_call(64, 32, 8, 128, 16, 256, 0, pa.PA_FP8_E4M3) == 2
    assert pa.pa_decode_kernels_per_call(256, 32, 32, 128, 16, 64, 0, pa.PA_FP8_E4M3) == 2
    try:
        for mode, want in ((1, 1), (2, 2)):
            pa.pa_debug_set_merge_mode(mode)
            assert pa.pa_decode_kernels_per_call(64, 32, 8, 128, 16, 64, 0, pa.PA_BF16) == want
            assert pa.pa_decode_kernels_per_call(64, 32, 8, 128, 16, 64, 0, pa.PA_F32) == 2
    finally:
        pa.pa_debug_set_merge_mode(0)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [("bf16", 32, 8, 128, 16), ("bf16", 8, 8, 128, 16),
                                               ("bf16", 16, 2, 64, 32), ("f32", 8, 2, 128, 16)])
def test_merge_modes_agree_bit_for_bit(dtype, hq, hkv, d, bs):
    """The in-kernel merge (by whichever CTA completes a segment, mid-range or after its range)
    and the merge kernel fold the pieces in the same order with the same arithmetic."""
    import paged_kv_cache_280_gb300 as pa

    w = W.random_case(41 + hq, 40, hq, hkv, d, bs, dtype, max_len=1500, min_len=1)
    c = DecodeCase(w).device()
    outs = []
    try:
        pa.pa_decode_set_ctas_per_sm(8)
        for mode in (1, 2, 1):
            pa.pa_debug_set_merge_mode(mode)
            c.dout.fill_(float("nan"))
            ws = c.run()
            outs.append(to_numpy(c.dout).copy())
            assert status_word(ws) == 0
    finally:
        pa.pa_decode_set_ctas_per_sm(0)
        pa.pa_debug_set_merge_mode(0)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    check_close(outs[0], c.oracle(), dtype)


def test_more_ctas_than_tiles():
    w = W.random_case(8, 3, 8, 8, 64, 16, "f32", max_len=20, min_len=1)
    c = DecodeCase(w).device()
    c.run()
    check_close(to_numpy(c.dout), c.oracle(), "f32")


@pytest.mark.parametrize("merge", [1, 2])
@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [("bf16", 8, 2, 128, 16), ("f32", 2, 2, 64, 16)])
def test_empty_ranges_and_long_merges(dtype, hq, hkv, d, bs, merge):
    """Runs of empty sequences between long ones, at 8 CTAs per SM over a few hundred
    tiles.  Without partitions the ranges balance tiles plus a fixed cost per segment, so
    ranges that fall in the gap before a segment are empty; long segments split into
    pieces of a tile or two, 40 and more per segment, all merged by one warp."""
    import paged_kv_cache_280_gb300 as pa

    w = W.random_case(31 + hq, 24, hq, hkv, d, bs, dtype, max_len=700, min_len=1)
    lens = np.zeros(24, np.int32)
    lens[[3, 9, 10, 17, 23]] = [700, 1, 333, 16 * 40, 47]
    c = DecodeCase(w, lengths=lens).device()
    ref = c.oracle()
    try:
        pa.pa_decode_set_ctas_per_sm(8)
        pa.pa_debug_set_merge_mode(merge)
        ws = c.run()
        first = to_numpy(c.dout).copy()
        c.dout.fill_(float("nan"))
        c.run(ws=ws)
        assert np.array_equal(first, to_numpy(c.dout))
    finally:
        pa.pa_decode_set_ctas_per_sm(0)
        pa.pa_debug_set_merge_mode(0)
    check_close(first, ref, dtype)
    assert status_word(ws) == 0
    assert not first[lens == 0].any()


def test_all_sequences_empty():
    w = W.random_case(9, 5, 4, 1, 64, 16, "bf16", max_len=0)
    c = DecodeCase(w, max_blocks=2).device()
    c.dout.fill_(1.0)
    ws = c.run(max_seq_len=32)
    assert not to_numpy(c.dout).any() and status_word(ws) == 0


def test_bad_table_entry_is_flagged_not_faulted():
    import torch

    w = W.random_case(10, 4, 8, 2, 128, 16, "bf16", max_len=200, min_len=40)
    c = DecodeCase(w).device()
    tables = c.tables.copy()
    tables[2, 1] = w.num_blocks + 5  # outside the pool
    c.dtables = to_torch(tables)
    ws = c.run()
    assert status_word(ws) & 1  # PA_DEV_BAD_BLOCK_ID
    ok = [0, 1, 3]
    check_close(to_numpy(c.dout), c.oracle(seqs=ok), "bf16", rows=ok)
    assert torch.isfinite(c.dout.float()).all()


def test_bad_seq_len_is_flagged_and_clamped():
    w = W.random_case(11, 3, 4, 4, 64, 16, "f32", max_len=60, min_len=10)
    c = DecodeCase(w).device()
    lens = c.lengths.copy()
    lens[1] = -5
    c.dlens = to_torch(lens)
    ws = c.run()
    assert status_word(ws) & 4  # PA_DEV_BAD_SEQ_LEN
    out = to_numpy(c.dout)
    assert not out[1].any()  # clamped to an empty sequence
    check_close(out, c.oracle(seqs=[0, 2]), "f32", rows=[0, 2])


def test_host_checks():
    import torch
    import paged_kv_cache_280_gb300 as pa

    w = W.random_case(12, 2, 4, 4, 64, 16, "bf16", max_len=40, min_len=1)
    c = DecodeCase(w).device()
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError) as e:
        c.run(ws=small)
    assert e.value.name == "PA_ERR_WORKSPACE_TOO_SMALL"
    with pytest.raises(pa.PAError) as e:
        c.run(partition_tokens=24)  # not a multiple of the block size
    assert e.value.name == "PA_ERR_INVALID_ARG"
    with pytest.raises(pa.PAError) as e:
        q9 = torch.zeros(2, 36, 64, dtype=torch.bfloat16, device="cuda")  # 9 query heads per KV head
        pa.pa_decode_attention(torch.empty_like(q9), q9, c.dk, c.dv, c.dtables, c.dlens, 40, 0.1, c.workspace())
    assert e.value.name == "PA_ERR_UNSUPPORTED"


def test_gqa4_batch64_full():
    """The bf16 GQA-4 batch of 64 skew-mixed lengths (32/8 heads, d 128): every output element."""
    c = DecodeCase(W.gqa4_b64()).device()
    ws = c.run()
    check_close(to_numpy(c.dout), c.oracle(), "bf16")
    assert status_word(ws) == 0


def test_launch_info():
    import paged_kv_cache_280_gb300 as pa

    ctas, stages, smem, mma = pa.pa_decode_launch_info(64, 32, 8, 128, 16, 256, pa.PA_BF16)
    # a stage of the tensor-core path holds two 16-token tiles (16 KB of K and V); the ring holds two
    assert mma == 1 and stages >= 2 and ctas >= 1 and smem > 32 * 1024
    ctas, stages, smem, mma = pa.pa_decode_launch_info(4, 4, 4, 64, 16, 3, pa.PA_F32)
    assert mma == 0 and ctas <= 4 * 4 * 3


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", VARIANTS)
def test_variants_ignore_nan_in_unused_slots(dtype, hq, hkv, d, bs):
    """Free blocks and the unfilled tail of each last block hold NaN; no output may see them."""
    w = W.random_case(700 + hq + d + bs, 9, hq, hkv, d, bs, dtype, max_len=200)
    lens = w.lengths.copy()
    lens[:4] = [1, bs - 1, bs + 1, 3 * bs - 5]
    c = DecodeCase(w, lengths=lens)
    assert poison_unused_slots(c.k_pool, c.v_pool, c.ref_tables, c.lengths) > 0
    c.device()
    ws = c.run()
    check_close(to_numpy(c.dout), c.oracle(), dtype)
    assert status_word(ws) == 0
