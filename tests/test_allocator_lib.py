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
