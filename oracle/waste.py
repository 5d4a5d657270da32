"""ORACLE -- test infrastructure only.  Memory accounting of the waste simulation.

Restates (not copies) the accounting of "用模拟把浪费率算出来" on the
ohmygp.com page: N requests either each reserve MAX_LEN contiguous slots,
or take ceil(len / BLOCK) blocks of BLOCK slots on demand.
  reserved waste = 1 - sum(len) / (N * MAX_LEN)
  paged waste    = 1 - sum(len) / sum(ceil(len / BLOCK) * BLOCK)
  concurrency    = (N * MAX_LEN) / sum(ceil(len / BLOCK) * BLOCK)
"""
from __future__ import annotations


def simulate(lengths, max_len=4096, block=16):
    used = 0
    reserved = 0
    paged = 0
    for n in lengths:
        n = int(n)
        used += n
        reserved += max_len
        paged += -(-n // block) * block
    return {
        "reserved_waste": 1.0 - used / reserved,
        "paged_waste": 1.0 - used / paged,
        "concurrency": reserved / paged,
        "used": used,
        "reserved": reserved,
        "paged": paged,
    }
