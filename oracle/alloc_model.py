"""ORACLE -- test infrastructure only.  Reference model of the block allocator.

Written from the pages' description, independently of the library's C++
allocator:

* On-demand blocks ("Q32" page §2 非连续存储; ohmygp.com 按需分配): a
  sequence takes a new physical block only when its tail block is full;
  existing KV never moves.
* Block table (same §2 Block Table映射; ohmygp.com 块表映射): logical block
  i of a sequence -> physical block id; the token at position t lives in
  slot ``table[t // bs] * bs + t % bs``.
* Refcounted sharing and copy-on-write ("Q32" §3; data.6616ai.com
  "Copy-on-write 共享"; ohmygp.com 写时共享): forked sequences point at
  the same physical blocks and each block counts its sharers; a sequence
  that writes a new token into a block whose refcount is above 1 first gets
  a private copy of it.

Readings of points the pages leave open (the same readings the library
follows, stated here so the model can be checked by eye):

* Free list: a FIFO queue whose initial order is given (a seeded
  permutation in the workloads); allocation pops the front, a freed block
  is pushed at the back.
* Copy-on-write trigger: at a sequence's write into its tail block, if the
  tail's refcount is above 1: take a fresh block n, emit the pair
  (tail, n), decrement the tail's refcount, set refcount[n] = 1 and point
  the table entry at n.  The last remaining sharer therefore writes in
  place, and a full shared block (never written again) is never copied.
* Fork copies the parent's table and length and adds one reference to each
  of its blocks; free walks the table in logical order, dropping one
  reference per block and returning blocks that reach zero.
* A batch append processes its sequence ids in the order given.
* Every call is all-or-nothing: on failure the state is unchanged.
* Swap-out of a preempted sequence (data.6616ai.com "PagedAttention 之外":
  KV swapped to CPU memory when memory is short, restored to resume):
  swap-out reports the table and then drops the sequence's references as
  free does, keeping its id and length; the sequence then takes no appends,
  forks or table reads.  Swap-in takes ceil(len / bs) fresh blocks from the
  front of the free list (refcount 1 each), which become its table.
"""
from __future__ import annotations

import copy
from collections import deque


class AllocError(Exception):
    code = "error"


class OutOfBlocks(AllocError):
    code = "out_of_blocks"


class NoSuchSeq(AllocError):
    code = "no_such_seq"


class SeqExists(AllocError):
    code = "seq_exists"


class RefcountLimit(AllocError):
    code = "refcount_limit"


class SeqSwapped(AllocError):
    code = "seq_swapped"


class RefAllocator:
    def __init__(self, num_blocks, block_size, free_order=None, max_refcount=0):
        if free_order is None:
            free_order = range(num_blocks)
        free_order = [int(b) for b in free_order]
        assert sorted(free_order) == list(range(num_blocks)), "free order must be a permutation"
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.max_refcount = int(max_refcount)
        self.free = deque(free_order)
        self.ref = [0] * self.num_blocks
        self.tables = {}
        self.lens = {}
        self.swapped = set()
        self.cow_copies = 0

    # -- helpers -----------------------------------------------------------
    def _take(self):
        if not self.free:
            raise OutOfBlocks()
        b = self.free.popleft()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _append_one(self, sid, slots, pairs):
        table = self.tables[sid]
        n = self.lens[sid]
        bs = self.block_size
        if n % bs == 0:
            table.append(self._take())
        else:
            tail = table[-1]
            if self.ref[tail] > 1:
                fresh = self._take()
                pairs.append((tail, fresh))
                self.ref[tail] -= 1
                table[-1] = fresh
                self.cow_copies += 1
        slots.append(table[n // bs] * bs + n % bs)
        self.lens[sid] = n + 1

    def _transaction(self, fn):
        saved = (copy.copy(self.free), list(self.ref), {k: list(v) for k, v in self.tables.items()},
                 dict(self.lens), self.cow_copies)
        try:
            return fn()
        except AllocError:
            self.free, self.ref, self.tables, self.lens, self.cow_copies = saved
            raise

    # -- API ---------------------------------------------------------------
    def create(self, sid):
        if sid in self.tables:
            raise SeqExists()
        self.tables[sid] = []
        self.lens[sid] = 0

    def _live(self, sid):
        if sid not in self.tables:
            raise NoSuchSeq()
        if sid in self.swapped:
            raise SeqSwapped()

    def append(self, sid, n_tokens):
        """Append n_tokens to one sequence; returns (slots, cow_pairs)."""
        self._live(sid)

        def run():
            slots, pairs = [], []
            for _ in range(n_tokens):
                self._append_one(sid, slots, pairs)
            return slots, pairs

        return self._transaction(run)

    def append_batch(self, sids):
        """One token for each id, in order; returns (slots, cow_pairs)."""
        for sid in sids:
            self._live(sid)

        def run():
            slots, pairs = [], []
            for sid in sids:
                self._append_one(sid, slots, pairs)
            return slots, pairs

        return self._transaction(run)

    def fork(self, parent, child):
        self._live(parent)
        if child in self.tables:
            raise SeqExists()
        table = self.tables[parent]
        if self.max_refcount > 0:
            for b in table:
                if self.ref[b] + 1 > self.max_refcount:
                    raise RefcountLimit()
        for b in table:
            self.ref[b] += 1
        self.tables[child] = list(table)
        self.lens[child] = self.lens[parent]

    def free_seq(self, sid):
        if sid not in self.tables:
            raise NoSuchSeq()
        for b in self.tables[sid]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.tables[sid]
        del self.lens[sid]
        self.swapped.discard(sid)

    def swap_out(self, sid):
        """Drop the sequence's blocks (as free does) but keep it; returns the table to copy out."""
        self._live(sid)
        table = self.tables[sid]
        for b in table:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        self.tables[sid] = []
        self.swapped.add(sid)
        return list(table)

    def swap_in(self, sid):
        """Fresh private blocks for a swapped-out sequence; returns them (its new table)."""
        if sid not in self.tables:
            raise NoSuchSeq()
        if sid not in self.swapped:
            raise AllocError()
        need = -(-self.lens[sid] // self.block_size)
        if need > len(self.free):
            raise OutOfBlocks()
        self.tables[sid] = [self._take() for _ in range(need)]
        self.swapped.discard(sid)
        return list(self.tables[sid])

    def table(self, sid):
        self._live(sid)
        return list(self.tables[sid])

    def length(self, sid):
        return self.lens[sid]

    def refcount(self, blk):
        return self.ref[blk]

    def free_list(self):
        return list(self.free)

    def stats(self):
        used = sum(1 for r in self.ref if r > 0)
        tokens = sum(self.lens.values())
        return {
            "num_blocks": self.num_blocks,
            "free_blocks": len(self.free),
            "used_blocks": used,
            "num_seqs": len(self.tables),
            "tokens": tokens,
            "slots": used * self.block_size,
            "shared_blocks": sum(1 for r in self.ref if r > 1),
            "cow_copies": self.cow_copies,
        }


def tail_waste(length, block_size):
    """Unused slots of a sequence: only its last block can be partly empty."""
    return -(-length // block_size) * block_size - length
