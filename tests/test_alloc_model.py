"""Pins of the allocator reference model: page facts, a hand-computed trace and invariants."""
import random

import pytest

from golden_io import lines, table
from oracle.alloc_model import OutOfBlocks, RefAllocator, RefcountLimit, SeqExists, NoSuchSeq, tail_waste


def run_trace(make_alloc, name="alloc_trace.txt"):
    """Replay tests/golden/alloc_trace.txt against an allocator object; returns it."""
    g, seq = table(name)
    a = make_alloc(int(g["num_blocks"][0]), int(g["block_size"][0]), [int(x) for x in g["free_order"]])
    last = None
    for parts in seq:
        key = parts[0]
        if key == "op":
            op, args = parts[1], [int(x) for x in parts[2:]]
            if op == "create":
                a.create(args[0])
            elif op == "append":
                last = a.append(args[0], args[1])
            elif op == "append_batch":
                last = a.append_batch(args)
            elif op == "fork":
                a.fork(args[0], args[1])
            elif op == "free":
                a.free_seq(args[0])
        elif key == "expect":
            what, vals = parts[1], [int(x) for x in parts[2:]]
            if what == "slots":
                assert list(last[0]) == vals
            elif what == "pairs":
                assert [tuple(p) for p in last[1]] == [tuple(vals[i:i + 2]) for i in range(0, len(vals), 2)]
            elif what == "refcount":
                assert a.refcount(vals[0]) == vals[1]
        elif key == "final":
            what, vals = parts[1], [int(x) for x in parts[2:]]
            if what == "table":
                assert a.table(vals[0]) == vals[1:]
            elif what == "len":
                assert a.length(vals[0]) == vals[1]
            elif what == "refcount":
                assert a.refcount(vals[0]) == vals[1]
            elif what == "free":
                assert a.free_list() == vals
            elif what == "cow_copies":
                assert a.stats()["cow_copies"] == vals[0]
    return a


def test_page_mapping_example():
    # logical 0 -> physical 5, logical 1 -> physical 12 (page 1, Block Table映射)
    parts = list(lines("mapping_example.txt"))
    bs = int(parts[0][1])
    tbl = [int(x) for x in parts[1][1:]]
    a = RefAllocator(16, bs, free_order=tbl + [b for b in range(16) if b not in tbl])
    a.create(0)
    slots, pairs = a.append(0, 32)
    assert a.table(0) == tbl and pairs == []
    for p in parts[2:]:
        assert slots[int(p[1])] == int(p[2])


def test_block32_tail_waste_example():
    parts = list(lines("block32_example.txt"))
    n = int(parts[0][1])
    for p in parts[1:]:
        bs, slots, wasted = int(p[1]), int(p[2]), int(p[3])
        a = RefAllocator(8, bs)
        a.create(0)
        a.append(0, n)
        assert a.stats()["slots"] == slots
        assert tail_waste(n, bs) == wasted == slots - n


def test_scripted_trace():
    run_trace(lambda nb, bs, order: RefAllocator(nb, bs, free_order=order))


def test_out_of_blocks_leaves_state_unchanged():
    a = RefAllocator(2, 16, free_order=[1, 0])
    a.create(0)
    a.append(0, 5)
    before = (a.free_list(), a.table(0), a.length(0), [a.refcount(b) for b in range(2)])
    with pytest.raises(OutOfBlocks):
        a.append(0, 40)  # needs two more blocks, one is free
    assert before == (a.free_list(), a.table(0), a.length(0), [a.refcount(b) for b in range(2)])
    a.create(1)
    a.fork(0, 2)
    with pytest.raises(OutOfBlocks):
        a.append_batch([1, 2, 0])  # 1 needs a block (ok), 2 needs a CoW block (none left)
    assert a.table(1) == [] and a.length(2) == 5 and a.free_list() == [0]


def test_errors():
    a = RefAllocator(4, 16)
    a.create(1)
    with pytest.raises(SeqExists):
        a.create(1)
    with pytest.raises(NoSuchSeq):
        a.append(2, 1)
    with pytest.raises(NoSuchSeq):
        a.fork(2, 3)
    a.append(1, 3)
    b = RefAllocator(4, 16, max_refcount=2)
    b.create(0)
    b.append(0, 1)
    b.fork(0, 1)
    with pytest.raises(RefcountLimit):
        b.fork(0, 2)


@pytest.mark.parametrize("writers", [8, 5, 1])
def test_cow_counts_for_parallel_sampling(writers):
    """A prompt of 1031 tokens shared by 8 samples: only the partial tail block is ever copied.

    If every sample writes, the first 7 copy and the last writes in place; if
    fewer write, every writer copies (the silent samples keep their reference).
    """
    a = RefAllocator(200, 16, free_order=list(range(200)))
    a.create(0)
    a.append(0, 1031)
    for s in range(8):
        a.fork(0, 1 + s)
    a.free_seq(0)
    assert all(a.refcount(b) == 8 for b in a.table(1))
    slots, pairs = a.append_batch([1 + s for s in range(writers)])
    want = 7 if writers == 8 else writers
    assert len(pairs) == want
    tail = a.table(8 if writers == 8 else 1)  # any table that still shares the full blocks
    assert all(p[0] == 64 for p in pairs)  # the partial block (physical 64 = logical 64) is the source
    full_blocks = a.table(1)[:64]
    assert all(a.refcount(b) == 8 for b in full_blocks)  # full shared blocks never copied
    assert tail[:64] == full_blocks


def _check_invariants(a):
    holders = {}
    for sid, tbl in a.tables.items():
        for b in tbl:
            holders[b] = holders.get(b, 0) + 1
        assert len(tbl) == -(-a.length(sid) // a.block_size)
        assert 0 <= tail_waste(a.length(sid), a.block_size) < a.block_size
    for b in range(a.num_blocks):
        assert a.refcount(b) == holders.get(b, 0)
    free = a.free_list()
    assert len(set(free)) == len(free)
    assert set(free) == {b for b in range(a.num_blocks) if a.refcount(b) == 0}
    assert len(free) + len(holders) == a.num_blocks


@pytest.mark.parametrize("seed", range(6))
def test_random_traces_keep_invariants(seed):
    rnd = random.Random(seed)
    a = RefAllocator(64, rnd.choice([4, 16]), free_order=rnd.sample(range(64), 64))
    live, nxt = [], 0
    for _ in range(400):
        op = rnd.random()
        try:
            if op < 0.15 or not live:
                a.create(nxt)
                live.append(nxt)
                nxt += 1
            elif op < 0.55:
                sid = rnd.choice(live)
                tail = a.table(sid)[-1] if a.table(sid) else None
                shared = tail is not None and a.refcount(tail) > 1 and a.length(sid) % a.block_size
                slots, pairs = a.append(sid, rnd.randint(1, 20))
                # copy only when writing into a shared, partly filled tail
                assert len(pairs) == (1 if shared else 0)
            elif op < 0.75:
                ids = rnd.sample(live, min(len(live), rnd.randint(1, 5)))
                a.append_batch(ids)
                # no sequence ever holds a shared block that it could still write into
            elif op < 0.88:
                parent = rnd.choice(live)
                a.fork(parent, nxt)
                live.append(nxt)
                nxt += 1
            else:
                sid = rnd.choice(live)
                a.free_seq(sid)
                live.remove(sid)
        except OutOfBlocks:
            pass
        _check_invariants(a)


def test_model_swap_golden_trace():
    """The same hand-computed swap trace on the reference model."""
    from oracle.alloc_model import AllocError, OutOfBlocks, RefAllocator, SeqSwapped

    a = RefAllocator(6, 4, free_order=[5, 2, 0, 4, 1, 3])
    a.create(0)
    a.append(0, 6)
    a.fork(0, 1)
    assert a.swap_out(1) == [5, 2]
    assert (a.refcount(5), a.refcount(2)) == (1, 1) and a.free_list() == [0, 4, 1, 3]
    with pytest.raises(SeqSwapped):
        a.append(1, 1)
    assert a.swap_out(0) == [5, 2] and a.free_list() == [0, 4, 1, 3, 5, 2]
    assert a.swap_in(1) == [0, 4] and a.length(1) == 6 and a.refcount(0) == 1
    slots, pairs = a.append(1, 1)
    assert slots == [18] and pairs == []
    with pytest.raises(AllocError):
        a.swap_in(1)
    a.create(2)
    a.append(2, 16)
    with pytest.raises(OutOfBlocks):
        a.swap_in(0)
    a.free_seq(0)
    assert a.stats()["num_seqs"] == 2
