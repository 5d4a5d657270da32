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
* Prefix caching (data.6616ai.com, paging's second dividend: blocks of a
  prefix common to many requests are cached and reused, so prefill computes
  only the rest): a full block is identified by the token ids of the whole
  prefix it completes.  Registering a sequence's first n tokens records its
  first n // bs full blocks (a prefix already recorded, or a block already
  recorded, keeps its entry).  A new sequence created from a prompt of n
  tokens starts with the longest run of recorded blocks matching the prompt,
  at most (n - 1) // bs of them (one prompt token is always left to compute),
  each taking one more reference; its length is the tokens they cover.  A
  recorded block whose last reference goes is not freed but kept, evictable;
  allocation takes the free list first, then evicts the block released
  longest ago (dropping its record).
"""
from __future__ import annotations

import copy
from collections import OrderedDict, deque


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
        self.prefix = {}               # token prefix (tuple) -> the block completing it
        self.cached = {}               # recorded block -> its prefix
        self.evictable = OrderedDict()  # recorded blocks with no reference, oldest release first

    # -- helpers -----------------------------------------------------------
    def _take(self):
        if self.free:
            b = self.free.popleft()
        elif self.evictable:
            b, _ = self.evictable.popitem(last=False)
            del self.prefix[self.cached.pop(b)]
        else:
            raise OutOfBlocks()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _release(self, b):
        """The block's last reference went: a recorded block stays recorded (evictable), others are freed."""
        if b in self.cached:
            self.evictable[b] = True
        else:
            self.free.append(b)

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
                 dict(self.lens), self.cow_copies, dict(self.prefix), dict(self.cached), OrderedDict(self.evictable))
        try:
            return fn()
        except AllocError:
            (self.free, self.ref, self.tables, self.lens, self.cow_copies, self.prefix, self.cached,
             self.evictable) = saved
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
                self._release(b)
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
                self._release(b)
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
        if need > len(self.free) + len(self.evictable):
            raise OutOfBlocks()
        self.tables[sid] = [self._take() for _ in range(need)]
        self.swapped.discard(sid)
        return list(self.tables[sid])

    def create_cached(self, sid, tokens):
        """Create a sequence starting with the longest recorded run of full blocks of ``tokens``."""
        if sid in self.tables:
            raise SeqExists()
        bs, tokens = self.block_size, [int(t) for t in tokens]
        hits = []
        for i in range(max(0, (len(tokens) - 1) // bs)):
            b = self.prefix.get(tuple(tokens[: (i + 1) * bs]))
            if b is None or (self.max_refcount > 0 and self.ref[b] + 1 > self.max_refcount):
                break
            hits.append(b)
        for b in hits:
            self.evictable.pop(b, None)
            self.ref[b] += 1
        self.tables[sid] = hits
        self.lens[sid] = len(hits) * bs
        return len(hits) * bs

    def cache_prefix(self, sid, tokens):
        """Record the full blocks of the sequence's first len(tokens) tokens."""
        self._live(sid)
        bs, tokens = self.block_size, [int(t) for t in tokens]
        if len(tokens) > self.lens[sid]:
            raise AllocError()
        for i in range(len(tokens) // bs):
            key, b = tuple(tokens[: (i + 1) * bs]), self.tables[sid][i]
            if key not in self.prefix and b not in self.cached:
                self.prefix[key] = b
                self.cached[b] = key

    def prefix_cache_stats(self):
        return {"cached_blocks": len(self.cached), "evictable_blocks": len(self.evictable)}

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
