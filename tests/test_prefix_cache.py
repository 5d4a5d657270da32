"""Prefix caching: the library allocator and the reference model against a hand-computed trace,
and against each other on randomized traces mixing cache operations with appends, forks, frees
and swaps."""
import random

import pytest

import paged_kv_cache_280_gb300 as pa
from oracle.alloc_model import OutOfBlocks, RefAllocator

T = [100 + i for i in range(16)]  # a prompt's token ids
U = [7] + T[1:]                   # differs in the first token


class Lib:
    def __init__(self, *a, **k):
        self.a = pa.Allocator(*a, **k)

    def __getattr__(self, name):
        return getattr(self.a, name)

    def append(self, sid, n):
        s, p = self.a.append(sid, n)
        return s.tolist(), [tuple(x) for x in p.tolist()]

    def append_batch(self, ids):
        s, p = self.a.append_batch(ids)
        return s.tolist(), [tuple(x) for x in p.tolist()]

    def swap_out(self, sid):
        return self.a.swap_out(sid).tolist()

    def swap_in(self, sid):
        return self.a.swap_in(sid).tolist()


@pytest.mark.parametrize("impl", [Lib, RefAllocator])
def test_golden_prefix_trace(impl):
    a = impl(6, 4, free_order=[5, 2, 0, 4, 1, 3])
    a.create(0)
    a.append(0, 9)                                   # blocks 5, 2, 0
    a.cache_prefix(0, T[:9])                         # records T[:4] -> 5, T[:8] -> 2 (block 0 is not full)
    assert a.prefix_cache_stats() == {"cached_blocks": 2, "evictable_blocks": 0}
    a.free_seq(0)                                    # 5, 2 stay cached (evictable), 0 is freed
    assert a.free_list() == [4, 1, 3, 0] and a.prefix_cache_stats()["evictable_blocks"] == 2
    assert a.create_cached(1, T[:10]) == 8           # at most (10 - 1) // 4 = 2 blocks: both hit, revived
    assert a.table(1) == [5, 2] and a.refcount(5) == 1 and a.prefix_cache_stats()["evictable_blocks"] == 0
    assert a.append(1, 2) == ([16, 17], [])          # token 8 starts a fresh block (4)
    assert a.create_cached(2, U[:10]) == 0           # first block differs: no hit
    assert a.create_cached(3, T[:5]) == 4 and a.refcount(5) == 2  # one block at most for 5 tokens
    assert a.create_cached(7, T[:8]) == 4            # 8 tokens: (8 - 1) // 4 = 1 block, one token left to compute
    a.free_seq(7)
    a.free_seq(1)                                    # 2 becomes evictable again, 4 is freed
    assert a.free_list() == [1, 3, 0, 4] and a.prefix_cache_stats()["evictable_blocks"] == 1
    a.create(4)
    a.append(4, 16)                                  # takes the whole free list
    assert a.table(4) == [1, 3, 0, 4] and a.free_list() == []
    a.create(5)
    assert a.append(5, 1) == ([8], [])               # free list empty: evicts 2, dropping T[:8]
    assert a.prefix_cache_stats() == {"cached_blocks": 1, "evictable_blocks": 0}
    assert a.create_cached(6, T[:9]) == 4 and a.refcount(5) == 2  # T[:4] still hits (held by 3 and 6); T[:8] is gone
    a.create(8)
    with pytest.raises((pa.PAError, OutOfBlocks)):
        a.append(8, 1)                               # nothing free, nothing evictable: all or nothing
    assert a.length(8) == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_prefix_traces_match_model(seed):
    rnd = random.Random(7000 + seed)
    nb, bs = rnd.choice([20, 48]), rnd.choice([2, 4])
    order = rnd.sample(range(nb), nb)
    lib, ref = Lib(nb, bs, free_order=order), RefAllocator(nb, bs, free_order=order)
    prompts = [[rnd.randint(0, 3) for _ in range(rnd.randint(1, 24))] for _ in range(6)]  # heavy sharing
    live, written, nxt = [], {}, 0  # written: tokens a sequence's KV holds, as far as the trace knows

    def both(fn):
        try:
            r = fn(ref)
        except OutOfBlocks:
            with pytest.raises(pa.PAError) as e:
                fn(lib)
            assert e.value.name == "PA_ERR_OUT_OF_BLOCKS"
            return False
        assert fn(lib) == r
        return True

    for _ in range(300):
        op = rnd.random()
        if op < 0.25 or not live:
            p = rnd.choice(prompts)
            n = ref.create_cached(nxt, p)
            assert lib.create_cached(nxt, p) == n
            live.append(nxt)
            written[nxt] = p[:n]
            if both(lambda a, s=nxt, k=len(p) - n: a.append(s, k)):
                written[nxt] = list(p)
            nxt += 1
        elif op < 0.45:
            sid = rnd.choice(live)
            w = written[sid]
            if w and len(w) == ref.length(sid):
                k = rnd.randint(0, len(w))
                lib.cache_prefix(sid, w[:k])
                ref.cache_prefix(sid, w[:k])
        elif op < 0.65:
            sid, k = rnd.choice(live), rnd.randint(1, 6)
            if both(lambda a: a.append(sid, k)):
                written[sid] = written[sid] + [rnd.randint(4, 9) for _ in range(k)]
        elif op < 0.75:
            parent = rnd.choice(live)
            lib.fork(parent, nxt)
            ref.fork(parent, nxt)
            live.append(nxt)
            written[nxt] = list(written[parent])
            nxt += 1
        else:
            sid = rnd.choice(live)
            lib.free_seq(sid)
            ref.free_seq(sid)
            live.remove(sid)
        assert lib.free_list() == ref.free_list()
        assert lib.prefix_cache_stats() == ref.prefix_cache_stats()
        for b in range(nb):
            assert lib.refcount(b) == ref.refcount(b)
        for sid in live:
            assert lib.table(sid) == ref.table(sid) and lib.length(sid) == ref.length(sid)
