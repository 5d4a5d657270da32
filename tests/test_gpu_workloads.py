"""GPU: the full-size workloads of the pages' shapes, in the launch configuration the benchmark uses.

* MHA batch of 256 skew-mixed lengths: one appended token per sequence
  (allocator -> slot-mapped append), then decode over len + 1.
* Parallel sampling: 16 prompts of 1031 tokens shared by 8 samples each,
  divergent tails U[0, 256]; copy-on-write pairs, pool contents after the
  copies and appends, and the decode of all 128 samples.
* 128K-token contexts (4 x 131072, 64/8 heads) with 2048-token partitions and
  with the balanced split, block sizes 16 and 32.
Large outputs are checked on sampled sequences the oracle computes one by one.
"""
import numpy as np
import pytest

import oracle
import synth.workloads as W
from gpu_cases import DecodeCase, check_close, status_word, to_numpy, to_torch
from oracle.alloc_model import RefAllocator

pytestmark = pytest.mark.gpu


def test_mha_b256_append_then_decode():
    import torch
    import paged_kv_cache_280_gb300 as pa

    w = W.mha_b256_append()
    B = w.num_seqs
    c = DecodeCase(w, max_blocks=int(-(-(int(w.lengths.max()) + 1) // 16)))
    slots, pairs = c.lib.append_batch(range(B))
    rslots, rpairs = c.ref.append_batch(list(range(B)))
    assert slots.tolist() == rslots and pairs.size == 0 and rpairs == []
    k_new, v_new = w.new_tokens("k", B), w.new_tokens("v", B)
    c.device()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(to_torch(k_new), to_torch(v_new), c.dk, c.dv, to_torch(slots), status=status)
    oracle.reshape_and_cache(k_new, v_new, c.k_pool, c.v_pool, slots)
    blk = torch.from_numpy(slots // 16).cuda()
    off = torch.from_numpy(slots % 16).cuda()
    got_k = to_numpy(c.dk[blk, :, off, :])
    got_v = to_numpy(c.dv[blk, :, off, :])
    assert np.array_equal(got_k, c.k_pool[slots // 16, :, slots % 16, :])
    assert np.array_equal(got_v, c.v_pool[slots // 16, :, slots % 16, :])
    assert status.item() == 0
    # decode over len + 1
    c.lengths = c.lengths + 1
    c.tables, lens = c.lib.export_tables(range(B), c.max_blocks)
    for s in range(B):
        t = c.ref.table(s)
        c.ref_tables[s, : len(t)] = t
    assert np.array_equal(c.tables, c.ref_tables) and lens.tolist() == c.lengths.tolist()
    c.dtables, c.dlens = to_torch(c.tables), to_torch(c.lengths)
    ws = c.run()
    order = np.argsort(c.lengths)
    sample = sorted(set(order[:4].tolist() + order[-4:].tolist() + list(range(0, B, 37))))
    check_close(to_numpy(c.dout), c.oracle(seqs=sample), "bf16", rows=sample)
    assert status_word(ws) == 0


def test_cow_parallel_sampling():
    import torch
    import paged_kv_cache_280_gb300 as pa

    w = W.cow_sampling()
    P, S, L, bs = w.prompts, w.samples, w.prompt_len, w.block_size
    order = w.free_order()
    lib = pa.Allocator(w.num_blocks, bs, free_order=order)
    ref = RefAllocator(w.num_blocks, bs, free_order=order.tolist())
    k_pool, v_pool = w.pool_values("k"), w.pool_values("v")
    dk, dv = to_torch(k_pool), to_torch(v_pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # prefill every prompt through the slot-mapped append
    prompt_slots = []
    for p in range(P):
        lib.create(p)
        ref.create(p)
        s_l, c_l = lib.append(p, L)
        s_r, c_r = ref.append(p, L)
        assert s_l.tolist() == s_r and c_l.size == 0
        prompt_slots.append(s_l)
    prompt_slots = np.concatenate(prompt_slots)
    pk, pv = w.prompt_tokens("k"), w.prompt_tokens("v")
    pa.pa_reshape_and_cache(to_torch(pk), to_torch(pv), dk, dv, to_torch(prompt_slots), status=status)
    oracle.reshape_and_cache(pk, pv, k_pool, v_pool, prompt_slots)
    # fork each prompt into its samples, then drop the prompt: every prompt block is shared 8 ways
    sid = lambda p, s: P + p * S + s  # noqa: E731
    for p in range(P):
        for s in range(S):
            lib.fork(p, sid(p, s))
            ref.fork(p, sid(p, s))
        lib.free_seq(p)
        ref.free_seq(p)
    assert all(lib.refcount(b) == S for b in lib.table(sid(0, 0)))
    # divergent tails, one decode step at a time, samples in order
    tails = w.tails()
    slots, pairs = [], []
    for t in range(int(tails.max())):
        ids = [sid(p, s) for p in range(P) for s in range(S) if tails[p * S + s] > t]
        s_l, c_l = lib.append_batch(ids)
        s_r, c_r = ref.append_batch(ids)
        assert s_l.tolist() == s_r and [tuple(x) for x in c_l.tolist()] == c_r
        slots.append(s_l)
        pairs.extend(c_r)
    slots = np.concatenate(slots)
    pairs = np.asarray(pairs, np.int32).reshape(-1, 2)
    # the pages' rule: only the partial prompt block is copied, once per writer except a last sole sharer
    total = 0
    for p in range(P):
        partial = int(prompt_slots[p * L + L - 1] // bs)
        writers = int((tails[p * S:(p + 1) * S] > 0).sum())
        expected = S - 1 if writers == S else writers
        assert sum(1 for a, _ in pairs.tolist() if a == partial) == expected
        total += expected
    assert len(pairs) == total  # no full shared block is ever copied
    k_new, v_new = w.new_tokens("k", len(slots)), w.new_tokens("v", len(slots))
    pa.pa_copy_blocks(dk, dv, to_torch(pairs), status=status)
    pa.pa_reshape_and_cache(to_torch(k_new), to_torch(v_new), dk, dv, to_torch(slots), status=status)
    oracle.copy_blocks(k_pool, v_pool, pairs)
    oracle.reshape_and_cache(k_new, v_new, k_pool, v_pool, slots)
    assert np.array_equal(to_numpy(dk), k_pool) and np.array_equal(to_numpy(dv), v_pool)
    assert status.item() == 0
    # decode all samples
    ids = [sid(p, s) for p in range(P) for s in range(S)]
    lens = (L + tails).astype(np.int32)
    max_blocks = int(-(-int(lens.max()) // bs))
    tables, got_lens = lib.export_tables(ids, max_blocks)
    assert got_lens.tolist() == lens.tolist()
    ref_tables = np.zeros_like(tables)
    for i, s in enumerate(ids):
        t = ref.table(s)
        ref_tables[i, : len(t)] = t
    assert np.array_equal(tables, ref_tables)
    q = w.queries()
    out = torch.empty(len(ids), w.num_q_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
    n = pa.pa_decode_workspace_bytes(len(ids), w.num_q_heads, w.num_kv_heads, w.head_dim)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    pa.pa_decode_attention(out, to_torch(q), dk, dv, to_torch(tables), to_torch(lens), int(lens.max()), w.scale, ws)
    ref_out = oracle.decode_attention(q, k_pool, v_pool, ref_tables, lens, w.scale, threads=8)
    check_close(to_numpy(out), ref_out, "bf16")
    assert int(ws[:4].view(torch.int32).item()) == 0


@pytest.mark.parametrize("bs", [16, 32])
def test_long_context_128k(bs):
    w = W.long_context(block_size=bs)
    c = DecodeCase(w).device()
    assert c.max_blocks == 131072 // bs
    sample = [0, 3]
    ref = c.oracle(seqs=sample, threads=2)
    ws = c.run(partition_tokens=2048)
    check_close(to_numpy(c.dout), ref, "bf16", rows=sample)
    assert status_word(ws) == 0
    c.dout.zero_()
    ws = c.run(ws=ws, partition_tokens=0)
    check_close(to_numpy(c.dout), ref, "bf16", rows=sample)
    assert status_word(ws) == 0
