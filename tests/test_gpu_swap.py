"""GPU: swap-out of preempted sequences to pinned host memory and swap-in to fresh blocks.

The stores must hold the pool's blocks bit for bit; after another sequence
has reused and overwritten the freed blocks, swapping back in must give a
decode output identical, bit for bit, to the one before the swap (same
lengths, so the same plan and arithmetic; only the physical ids differ).
"""
import numpy as np
import pytest

import synth.workloads as W
from gpu_cases import DecodeCase, to_numpy, to_torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [("bf16", 32, 8, 128, 16), ("f32", 8, 4, 64, 32), ("bf16", 16, 16, 64, 16)])
def test_swap_round_trip_is_bit_exact(dtype, hq, hkv, d, bs):
    import torch
    import paged_kv_cache_280_gb300 as pa

    w = W.random_case(900 + hq + d, 12, hq, hkv, d, bs, dtype, max_len=300, min_len=1, slack=1.6)
    c = DecodeCase(w).device()
    c.lib.fork(3, 50)  # sequence 3 shares its blocks: its swap-out must leave them with the sharer
    c.ref.fork(3, 50)
    c.run()
    before = to_numpy(c.dout).copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    stores = {}
    for s in (2, 3, 7):
        blocks = c.lib.swap_out(s)
        assert blocks.tolist() == c.ref.swap_out(s)
        n = len(blocks)
        kst = torch.empty((n, hkv, bs, d), dtype=tdt, pin_memory=True)
        vst = torch.empty((n, hkv, bs, d), dtype=tdt, pin_memory=True)
        bl = torch.from_numpy(blocks).pin_memory()
        pa.pa_swap_out(c.dk, c.dv, bl, kst, vst, status=status)
        stores[s] = (blocks, kst, vst)
    torch.cuda.synchronize()
    for s, (blocks, kst, vst) in stores.items():
        assert np.array_equal(to_numpy(kst), c.k_pool[blocks]) and np.array_equal(to_numpy(vst), c.v_pool[blocks])
    # the freed blocks (refcount 0 now) are anyone's: overwrite them with NaN; the shared ones stay live
    freed = [int(x) for blocks, _, _ in stores.values() for x in blocks if c.lib.refcount(int(x)) == 0]
    assert freed and all(c.lib.refcount(int(x)) == 1 for x in stores[3][0])
    idx = torch.tensor(freed, dtype=torch.long, device="cuda")
    c.dk[idx] = float("nan")
    c.dv[idx] = float("nan")
    # swap back in, to fresh private blocks
    for s, (_, kst, vst) in stores.items():
        blocks = c.lib.swap_in(s)
        assert blocks.tolist() == c.ref.swap_in(s)
        pa.pa_swap_in(kst, vst, torch.from_numpy(blocks).to("cuda"), c.dk, c.dv, status=status)
    tables, lens = c.lib.export_tables(range(len(c.lengths)), c.max_blocks)
    assert lens.tolist() == c.lengths.tolist()
    c.dtables = to_torch(tables)
    c.run()
    assert np.array_equal(to_numpy(c.dout), before)
    assert status.item() == 0
