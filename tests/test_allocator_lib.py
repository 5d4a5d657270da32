"""The library's C++ allocator against the oracle's reference model: bit-exact tables, slots,
copy-on-write pairs, refcounts and free-list order, plus the pages' waste figures."""
import math
import random

import numpy as np
import pytest

import paged_kv_cache_280_gb300 as pa
import synth
from oracle import waste
from oracle.alloc_model import OutOfBlocks, RefAllocator
from test_alloc_model import run_trace


class LibAdapter:
    """Exposes the library allocator through the reference model's method names."""

    def __init__(self, nb, bs, order, max_refcount=0):
        self.a = pa.Allocator(nb, bs, free_order=order, max_refcount=max_refcount)
        self.num_blocks, self.block_size = nb, bs
        self.tables = {}

    def create(self, sid):
        self.a.create(sid)
        self.tables[sid] = True

    def append(self, sid, n):
        s, p = self.a.append(sid, n)
        return s.tolist(), [tuple(x) for x in p.tolist()]

    def append_batch(self, sids):
        s, p = self.a.append_batch(sids)
        return s.tolist(), [tuple(x) for x in p.tolist()]

    def fork(self, p, c):
        self.a.fork(p, c)

    def free_seq(self, sid):
        self.a.free_seq(sid)

    def table(self, sid):
        return self.a.table(sid)

    def length(self, sid):
        return self.a.length(sid)

    def refcount(self, b):
        return self.a.refcount(b)

    def free_list(self):
        return self.a.free_list()

    def stats(self):
        return self.a.stats()


def test_golden_trace_on_library():
    run_trace(lambda nb, bs, order: LibAdapter(nb, bs, order))


def test_page_mapping_example_on_library():
    a = pa.Allocator(16, 16, free_order=[5, 12] + [b for b in range(16) if b not in (5, 12)])
    a.create(0)
    slots, pairs = a.append(0, 18)
    assert a.table(0) == [5, 12] and slots[17] == 193 and len(pairs) == 0


def _same_state(lib, ref, live):
    assert lib.free_list() == ref.free_list()
    for b in range(ref.num_blocks):
        assert lib.refcount(b) == ref.refcount(b)
    for sid in live:
        assert lib.table(sid) == ref.table(sid)
        assert lib.length(sid) == ref.length(sid)
    st = lib.stats()
    rs = ref.stats()
    for k in ("free_blocks", "used_blocks", "shared_blocks", "num_seqs", "tokens", "slots", "cow_copies"):
        assert st[k] == rs[k], k


@pytest.mark.parametrize("seed", range(8))
def test_random_traces_match_model(seed):
    rnd = random.Random(1000 + seed)
    nb = rnd.choice([16, 48, 96])
    bs = rnd.choice([4, 16, 32])
    order = rnd.sample(range(nb), nb)
    lib = pa.Allocator(nb, bs, free_order=order)
    ref = RefAllocator(nb, bs, free_order=order)
    live, nxt = [], 0
    for _ in range(300):
        op = rnd.random()
        if op < 0.12 or not live:
            lib.create(nxt)
            ref.create(nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.5:
            sid, n = rnd.choice(live), rnd.randint(0, 40)
            try:
                r = ref.append(sid, n)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as e:
                    lib.append(sid, n)
                assert e.value.name == "PA_ERR_OUT_OF_BLOCKS"
            else:
                s, p = lib.append(sid, n)
                assert s.tolist() == r[0] and [tuple(x) for x in p.tolist()] == r[1]
        elif op < 0.72:
            ids = [rnd.choice(live) for _ in range(rnd.randint(1, 6))]  # repeats allowed
            try:
                r = ref.append_batch(ids)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as e:
                    lib.append_batch(ids)
                assert e.value.name == "PA_ERR_OUT_OF_BLOCKS"
            else:
                s, p = lib.append_batch(ids)
                assert s.tolist() == r[0] and [tuple(x) for x in p.tolist()] == r[1]
        elif op < 0.86:
            parent = rnd.choice(live)
            lib.fork(parent, nxt)
            ref.fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        else:
            sid = rnd.choice(live)
            lib.free_seq(sid)
            ref.free_seq(sid)
            live.remove(sid)
        _same_state(lib, ref, live)


def test_errors_and_all_or_nothing():
    a = pa.Allocator(3, 16, free_order=[2, 0, 1], max_refcount=2)
    a.create(7)
    with pytest.raises(pa.PAError) as e:
        a.create(7)
    assert e.value.name == "PA_ERR_SEQ_EXISTS"
    with pytest.raises(pa.PAError) as e:
        a.append(8, 1)
    assert e.value.name == "PA_ERR_NO_SUCH_SEQ"
    a.append(7, 20)
    before = (a.free_list(), a.table(7), a.length(7))
    with pytest.raises(pa.PAError) as e:
        a.append(7, 40)  # needs 2 blocks, 1 free
    assert e.value.name == "PA_ERR_OUT_OF_BLOCKS"
    assert before == (a.free_list(), a.table(7), a.length(7))
    a.fork(7, 8)
    with pytest.raises(pa.PAError) as e:
        a.fork(7, 9)
    assert e.value.name == "PA_ERR_REFCOUNT_LIMIT"
    with pytest.raises(pa.PAError):
        pa.Allocator(4, 16, free_order=[0, 1, 1, 2])


def test_export_tables_layout():
    a = pa.Allocator(32, 16, free_order=synth.permutation(3, 32))
    for s, n in enumerate([0, 1, 16, 17, 70]):
        a.create(s)
        a.append(s, n)
    tables, lens = a.export_tables(range(5), 6)
    assert lens.tolist() == [0, 1, 16, 17, 70]
    for s in range(5):
        t = a.table(s)
        assert tables[s, : len(t)].tolist() == t and not tables[s, len(t):].any()
    with pytest.raises(pa.PAError) as e:
        a.export_tables(range(5), 4)
    assert e.value.name == "PA_ERR_BUFFER_TOO_SMALL"


def test_waste_simulation_through_library_allocator():
    """1000 requests of the pages' length mix: the library's paged accounting equals the oracle's,
    and lands within sampling error of the closed form (83.8 % reserved, 1.12 % paged, 6.10x)."""
    lens = synth.lengths_mix(synth.stream_seed(280000, 1), 1000)
    need = int(sum(-(-int(x) // 16) for x in lens))
    a = pa.Allocator(need, 16, free_order=synth.permutation(1, need))
    for s, n in enumerate(lens):
        a.create(s)
        a.append(s, int(n))
    st = a.stats()
    r = waste.simulate(lens, 4096, 16)
    assert st["slots"] == r["paged"] and st["tokens"] == r["used"] and st["free_blocks"] == 0
    paged_waste = 1 - st["tokens"] / st["slots"]
    assert paged_waste == pytest.approx(r["paged_waste"], abs=0)
    assert abs(r["reserved_waste"] - 0.83801) < 3 * 0.0058
    assert paged_waste < 0.04
    for s, n in enumerate(lens):  # waste only in the tail block
        assert 0 <= len(a.table(s)) * 16 - int(n) < 16


def test_outputs_in_place():
    """append_batch / export_tables write into caller arrays (pinned staging) exactly what they return."""
    order = list(range(40))[::-1]
    a = pa.Allocator(40, 16, free_order=order)
    b = pa.Allocator(40, 16, free_order=order)
    for s, n in enumerate([5, 16, 33]):
        for x in (a, b):
            x.create(s)
            x.append(s, n)
    a.fork(1, 9)
    b.fork(1, 9)
    ids = np.array([0, 1, 2, 9, 1], np.int64)
    slots = np.full(8, -7, np.int64)
    pairs = np.full((8, 2), -7, np.int32)
    s_in, p_in = a.append_batch(ids, slots_out=slots, pairs_out=pairs)
    s_ref, p_ref = b.append_batch(ids.tolist())
    assert s_in.tolist() == s_ref.tolist() and p_in.tolist() == p_ref.tolist()
    assert slots[:5].tolist() == s_ref.tolist() and slots[5:].tolist() == [-7] * 3
    tables = np.zeros((4, 5), np.int32)
    lens = np.zeros(4, np.int32)
    a.export_tables([0, 1, 2, 9], 5, tables_out=tables, lens_out=lens)
    t_ref, l_ref = b.export_tables([0, 1, 2, 9], 5)
    assert np.array_equal(tables, t_ref) and np.array_equal(lens, l_ref)
    with pytest.raises(ValueError):
        a.append_batch([0], slots_out=np.zeros(4, np.int32))
    with pytest.raises(ValueError):
        a.export_tables([0], 5, tables_out=np.zeros((1, 4), np.int32), lens_out=np.zeros(1, np.int32))


@pytest.mark.parametrize("seed", range(6))
def test_random_traces_with_swaps_match_model(seed):
    """Appends, forks, frees and swap-outs/ins interleaved: the library and the model stay identical."""
    from oracle.alloc_model import SeqSwapped

    rnd = random.Random(5000 + seed)
    nb, bs = rnd.choice([24, 64]), rnd.choice([4, 16])
    order = rnd.sample(range(nb), nb)
    lib = pa.Allocator(nb, bs, free_order=order)
    ref = RefAllocator(nb, bs, free_order=order)
    live, swapped, nxt = [], set(), 0

    def same_error(fn_lib, fn_ref):
        try:
            r = fn_ref()
        except OutOfBlocks:
            with pytest.raises(pa.PAError) as e:
                fn_lib()
            assert e.value.name == "PA_ERR_OUT_OF_BLOCKS"
            return None
        return r, fn_lib()

    for _ in range(400):
        op = rnd.random()
        active = [s for s in live if s not in swapped]
        if op < 0.1 or not live:
            lib.create(nxt)
            ref.create(nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.45 and active:
            sid, n = rnd.choice(active), rnd.randint(0, 20)
            out = same_error(lambda: lib.append(sid, n), lambda: ref.append(sid, n))
            if out:
                (rs, rp), (ls, lp) = out
                assert ls.tolist() == rs and [tuple(x) for x in lp.tolist()] == rp
        elif op < 0.6 and active:
            parent = rnd.choice(active)
            lib.fork(parent, nxt)
            ref.fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.75 and active:
            sid = rnd.choice(active)
            assert lib.swap_out(sid).tolist() == ref.swap_out(sid)
            swapped.add(sid)
        elif op < 0.9 and swapped:
            sid = rnd.choice(sorted(swapped))
            out = same_error(lambda: lib.swap_in(sid), lambda: ref.swap_in(sid))
            if out:
                assert out[1].tolist() == out[0]
                swapped.discard(sid)
        elif live:
            sid = rnd.choice(live)
            lib.free_seq(sid)
            ref.free_seq(sid)
            live.remove(sid)
            swapped.discard(sid)
        # state: free list, refcounts, tables of active sequences, lengths of all
        assert lib.free_list() == ref.free_list()
        for b in range(nb):
            assert lib.refcount(b) == ref.refcount(b)
        for sid in live:
            assert lib.length(sid) == ref.length(sid)
            if sid in swapped:
                with pytest.raises(pa.PAError) as e:
                    lib.table(sid)
                assert e.value.name == "PA_ERR_SEQ_SWAPPED"
                with pytest.raises(SeqSwapped):
                    ref.table(sid)
            else:
                assert lib.table(sid) == ref.table(sid)


def test_swap_golden_trace():
    """A hand-computed swap trace: shared blocks survive a sharer's swap-out; swap-in takes fresh private blocks."""
    a = pa.Allocator(6, 4, free_order=[5, 2, 0, 4, 1, 3])
    a.create(0)
    a.append(0, 6)                       # blocks 5, 2 (slots 20..23, 8..9)
    a.fork(0, 1)                         # refcounts 5:2, 2:2
    assert a.swap_out(1).tolist() == [5, 2]
    assert (a.refcount(5), a.refcount(2)) == (1, 1) and a.free_list() == [0, 4, 1, 3]
    with pytest.raises(pa.PAError) as e:
        a.append(1, 1)
    assert e.value.name == "PA_ERR_SEQ_SWAPPED"
    assert a.swap_out(0).tolist() == [5, 2]
    assert a.free_list() == [0, 4, 1, 3, 5, 2]
    assert a.swap_in(1).tolist() == [0, 4] and a.length(1) == 6
    assert a.table(1) == [0, 4] and a.refcount(0) == 1 and a.free_list() == [1, 3, 5, 2]
    s, p = a.append(1, 1)                # private tail: written in place, no copy
    assert s.tolist() == [4 * 4 + 2] and p.size == 0
    with pytest.raises(pa.PAError) as e:
        a.swap_in(1)                     # not swapped out
    assert e.value.name == "PA_ERR_INVALID_ARG"
    a.create(2)
    a.append(2, 16)                      # takes 1, 3, 5, 2: the pool is full
    with pytest.raises(pa.PAError) as e:
        a.swap_in(0)
    assert e.value.name == "PA_ERR_OUT_OF_BLOCKS" and a.length(0) == 6
    a.free_seq(0)                        # a swapped-out sequence can be dropped
    assert a.stats()["num_seqs"] == 2
