"""Pins of the oracle's slot-mapped append and copy-on-write block copy.

The two are element copies whose meaning the pages fix:

* append ("破局思路", ohmygp.com: each new token takes one slot of the
  sequence's current block; "Q32: vLLM PagedAttention 原理" §2: a token is
  written into its block and no existing KV moves; same §2 item 2 gives the
  mapping example logical 0 -> physical 5, logical 1 -> physical 12);
* copy-on-write ("Q32" §3 Copy-on-Write, ohmygp.com 写时共享: a shared block
  is copied to a new physical block when one sharer writes into it).

Checked against things other than the oracle itself:

* hand-placed destinations from the page's mapping example (token 17 of the
  table [5, 12] sits in physical block 12 at offset 1), with every value
  distinct so that a wrong head, slot, block or tensor fails, and every other
  pool element left untouched;
* the pinned decode oracle reading back what the append wrote: a sequence
  appended token by token through the allocator model into a scattered pool
  must decode to brute-force attention over its never-paged K and V (scipy);
* copy-on-write end to end: fork, the copy, the child's write, then the
  child decodes to its own contiguous history and the parent to its own.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth
from golden_io import table
from oracle import alloc_model

SENT_K, SENT_V = -1.0, -2.0


def _marked(n_tokens, Hkv, D, base):
    """Token i, head h, element e holds base + 1000 i + 100 h + e (all distinct, exact in fp32 and bf16)."""
    i, h, e = np.meshgrid(np.arange(n_tokens), np.arange(Hkv), np.arange(D), indexing="ij")
    return (base + 1000 * i + 100 * h + e).astype(np.float32)


def _bf16_bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_append_mapping_example_places_every_head_and_tensor():
    g, seq = table("mapping_example.txt")
    bs = int(g["block_size"][0])
    assert [int(x) for x in g["table"]] == [5, 12]
    slot = {int(p[1]): int(p[2]) for p in seq if p[0] == "token"}
    Hkv, D, nb = 3, 4, 16
    kp = np.full((nb, Hkv, bs, D), SENT_K, np.float32)
    vp = np.full((nb, Hkv, bs, D), SENT_V, np.float32)
    toks = [17, 0, 31]  # physical block 12 offset 1, block 5 offset 0, block 12 offset 15
    kn, vn = _marked(3, Hkv, D, 1.0), _marked(3, Hkv, D, 50_000.0)
    oracle.reshape_and_cache(kn, vn, kp, vp, np.array([slot[t] for t in toks], np.int64))
    expect_k = np.full_like(kp, SENT_K)
    expect_v = np.full_like(vp, SENT_V)
    for i, (blk, off) in enumerate([(12, 1), (5, 0), (12, 15)]):
        for h in range(Hkv):
            expect_k[blk, h, off, :] = kn[i, h, :]
            expect_v[blk, h, off, :] = vn[i, h, :]
    assert np.array_equal(kp, expect_k)
    assert np.array_equal(vp, expect_v)
    # token 17: every head of K and V, element by element
    for h in range(Hkv):
        assert kp[12, h, 1].tolist() == [1000 * 0 + 100 * h + e + 1.0 for e in range(D)]
        assert vp[12, h, 1].tolist() == [1000 * 0 + 100 * h + e + 50_000.0 for e in range(D)]


@pytest.mark.parametrize("elem", ["f32", "bf16"])
def test_append_skips_padding_and_refuses_out_of_range(elem):
    bs, Hkv, D, nb = 16, 2, 8, 4
    mk = (lambda a: a) if elem == "f32" else _bf16_bits
    kp = mk(np.full((nb, Hkv, bs, D), SENT_K, np.float32))
    vp = mk(np.full((nb, Hkv, bs, D), SENT_V, np.float32))
    kn, vn = mk(_marked(2, Hkv, D, 1.0)), mk(_marked(2, Hkv, D, 7.0))
    before_k, before_v = kp.copy(), vp.copy()
    oracle.reshape_and_cache(kn, vn, kp, vp, np.array([-1, -5], np.int64))  # padding: nothing written
    assert np.array_equal(kp, before_k) and np.array_equal(vp, before_v)
    # slot 0 is a real slot (block 0, offset 0), unlike the negative padding slots
    oracle.reshape_and_cache(kn[:1], vn[:1], kp, vp, np.array([0], np.int64))
    assert np.array_equal(kp[0, :, 0], kn[0]) and np.array_equal(vp[0, :, 0], vn[0])
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(kn[:1], vn[:1], kp, vp, np.array([nb * bs], np.int64))


def test_append_then_decode_equals_brute_force_on_contiguous_history():
    """What the append writes, the (independently pinned) decode oracle reads back."""
    bs, Hkv, G, D, nb = 4, 3, 2, 8, 12
    Hq, n = Hkv * G, 19
    order = synth.permutation(synth.stream_seed(2801, 9), nb)
    alloc = alloc_model.RefAllocator(nb, bs, free_order=order)
    alloc.create(0)
    K = synth.normal(synth.stream_seed(2801, 1), n * Hkv * D, "f32").reshape(n, Hkv, D)
    V = synth.normal(synth.stream_seed(2801, 2), n * Hkv * D, "f32").reshape(n, Hkv, D)
    q = synth.normal(synth.stream_seed(2801, 3), Hq * D, "f32").reshape(1, Hq, D)
    kp = np.full((nb, Hkv, bs, D), np.nan, np.float32)
    vp = np.full((nb, Hkv, bs, D), np.nan, np.float32)
    for t in range(n):  # one decode step at a time, as the allocator hands out slots
        slots, pairs = alloc.append(0, 1)
        assert not pairs
        oracle.reshape_and_cache(K[t:t + 1], V[t:t + 1], kp, vp, np.array(slots, np.int64))
    bt = np.array([alloc.table(0)], np.int32)
    assert sorted(bt[0].tolist()) != bt[0].tolist() or nb < 3  # the blocks really are scattered
    out = oracle.decode_attention(q, kp, vp, bt, np.array([n], np.int32), 0.3)
    for h in range(Hq):
        g = h // G
        w = softmax(0.3 * (K[:, g, :].astype(np.float64) @ q[0, h].astype(np.float64)))
        np.testing.assert_allclose(out[0, h], w @ V[:, g, :].astype(np.float64), rtol=0, atol=1e-12)


@pytest.mark.parametrize("elem", ["f32", "bf16"])
def test_copy_blocks_whole_block_k_and_v(elem):
    bs, Hkv, D, nb = 4, 3, 8, 10
    vals_k = np.arange(nb * Hkv * bs * D, dtype=np.float32).reshape(nb, Hkv, bs, D)
    vals_v = -1.0 - vals_k
    mk = (lambda a: a) if elem == "f32" else _bf16_bits
    kp, vp = mk(vals_k.copy()), mk(vals_v.copy())
    k0, v0 = kp.copy(), vp.copy()
    oracle.copy_blocks(kp, vp, [(3, 7), (0, 5)])
    expect_k, expect_v = k0.copy(), v0.copy()
    for src, dst in [(3, 7), (0, 5)]:
        for h in range(Hkv):
            for s in range(bs):  # every slot, filled or not
                expect_k[dst, h, s, :] = k0[src, h, s, :]
                expect_v[dst, h, s, :] = v0[src, h, s, :]
    assert np.array_equal(kp, expect_k) and np.array_equal(vp, expect_v)
    # sources unchanged, and no block other than the destinations changed
    changed = sorted({int(b) for b in np.nonzero((kp != k0).any(axis=(1, 2, 3)) | (vp != v0).any(axis=(1, 2, 3)))[0]})
    assert changed == [5, 7]
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kp, vp, [(1, nb)])
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kp, vp, [(-1, 2)])


def test_cow_fork_copy_append_keeps_both_histories():
    """Fork a 6-token sequence (bs 4: one full and one partial shared block); the child's first write copies
    the partial block, the parent's next write lands in place.  Each then decodes to its own history."""
    bs, Hkv, D, nb = 4, 2, 8, 8
    order = synth.permutation(synth.stream_seed(2802, 9), nb)
    alloc = alloc_model.RefAllocator(nb, bs, free_order=order)
    seed = synth.stream_seed(2802, 1)
    hist = synth.normal(seed, 2 * 8 * Hkv * D, "f32").reshape(2, 8, Hkv, D)  # [K|V][token][h][d]
    kp = np.full((nb, Hkv, bs, D), np.nan, np.float32)
    vp = np.full((nb, Hkv, bs, D), np.nan, np.float32)
    alloc.create(0)
    slots, _ = alloc.append(0, 6)
    oracle.reshape_and_cache(hist[0, :6], hist[1, :6], kp, vp, np.array(slots, np.int64))
    alloc.fork(0, 1)
    child_new = synth.normal(synth.stream_seed(2802, 2), 2 * Hkv * D, "f32").reshape(2, 1, Hkv, D)
    slots, pairs = alloc.append(1, 1)
    assert len(pairs) == 1 and pairs[0][0] == alloc.table(0)[1]
    oracle.copy_blocks(kp, vp, pairs)
    oracle.reshape_and_cache(child_new[0], child_new[1], kp, vp, np.array(slots, np.int64))
    slots, pairs = alloc.append(0, 1)
    assert not pairs  # the parent is now the block's only holder: in place
    oracle.reshape_and_cache(hist[0, 6:7], hist[1, 6:7], kp, vp, np.array(slots, np.int64))
    q = synth.normal(synth.stream_seed(2802, 3), 2 * Hkv * D, "f32").reshape(2, Hkv, D)
    bt = np.zeros((2, 2), np.int32)
    bt[0], bt[1] = alloc.table(0), alloc.table(1)
    out = oracle.decode_attention(q, kp, vp, bt, np.array([7, 7], np.int32), 0.25)
    parent = hist[:, :7]
    child = np.concatenate([hist[:, :6], child_new], axis=1)
    for b, (Kc, Vc) in enumerate([(parent[0], parent[1]), (child[0], child[1])]):
        for h in range(Hkv):
            w = softmax(0.25 * (Kc[:, h].astype(np.float64) @ q[b, h].astype(np.float64)))
            np.testing.assert_allclose(out[b, h], w @ Vc[:, h].astype(np.float64), rtol=0, atol=1e-12)
