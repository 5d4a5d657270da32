"""Helpers of the GPU parity tests: build one seeded case for both sides and compare.

The CUDA side gets its block tables from the library allocator, the oracle
side from the reference allocator model; both start from the same seeded
free-list order and the tests assert the two agree bit for bit.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth.workloads as W
from oracle.alloc_model import RefAllocator

BF16_ATOL = 1e-2
BF16_RTOL = 1e-2
F32_ATOL = 1e-5


def to_torch(a: np.ndarray, device="cuda"):
    import torch

    if a.dtype == np.uint16:  # bf16 bit patterns
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_numpy(t) -> np.ndarray:
    import torch

    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def widen(a: np.ndarray) -> np.ndarray:
    """bf16 bits or fp32 values -> float64 (exact)."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def check_close(gpu: np.ndarray, ref: np.ndarray, dtype: str, rows=None):
    """Elementwise bound of the workload: fp32 |d| <= 1e-5; bf16 |d| <= 1e-2 + 1e-2 |ref|."""
    g = widen(gpu)
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - ref)
    if dtype == "f32":
        bound = np.full_like(ref, F32_ATOL)
    else:
        bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), (
        f"max |err| {err.max():.3e}, worst at {np.unravel_index(worst, err.shape)}: gpu {g.flat[worst]:.6f} "
        f"ref {ref.flat[worst]:.6f}"
    )
    return float(err.max())


class DecodeCase:
    """A decode batch: pools, queries and block tables for both sides."""

    def __init__(self, w: W.Workload, lengths=None, max_blocks=None):
        import paged_kv_cache_280_gb300 as pa

        self.w = w
        self.lengths = np.asarray(w.lengths if lengths is None else lengths, np.int32)
        order = w.free_order()
        self.lib = pa.Allocator(w.num_blocks, w.block_size, free_order=order)
        self.ref = RefAllocator(w.num_blocks, w.block_size, free_order=order.tolist())
        for s, n in enumerate(self.lengths):
            self.lib.create(s)
            self.ref.create(s)
            ls, lp = self.lib.append(s, int(n))
            rs, rp = self.ref.append(s, int(n))
            assert ls.tolist() == rs and lp.size == 0 and rp == []
        need = max(1, int(max(-(-int(x) // w.block_size) for x in self.lengths)) if len(self.lengths) else 1)
        self.max_blocks = max(need, max_blocks or 0)
        self.tables, lens = self.lib.export_tables(range(len(self.lengths)), self.max_blocks)
        assert lens.tolist() == self.lengths.tolist()
        self.ref_tables = np.zeros_like(self.tables)
        for s in range(len(self.lengths)):
            t = self.ref.table(s)
            self.ref_tables[s, : len(t)] = t
        assert np.array_equal(self.tables, self.ref_tables)
        self.k_pool = w.pool_values("k")
        self.v_pool = w.pool_values("v")
        self.q = w.queries()

    def device(self):
        import torch

        self.dk = to_torch(self.k_pool)
        self.dv = to_torch(self.v_pool)
        self.dq = to_torch(self.q)
        self.dtables = to_torch(self.tables)
        self.dlens = to_torch(self.lengths)
        self.dout = torch.empty_like(self.dq)
        return self

    def workspace(self):
        import paged_kv_cache_280_gb300 as pa
        import torch

        n = pa.pa_decode_workspace_bytes(len(self.lengths), self.w.num_q_heads, self.w.num_kv_heads, self.w.head_dim)
        return torch.zeros(n, dtype=torch.uint8, device="cuda")

    def run(self, ws=None, partition_tokens=None, max_seq_len=None):
        import paged_kv_cache_280_gb300 as pa

        ws = self.workspace() if ws is None else ws
        pt = self.w.partition_tokens if partition_tokens is None else partition_tokens
        msl = int(self.lengths.max(initial=0)) if max_seq_len is None else max_seq_len
        pa.pa_decode_attention(self.dout, self.dq, self.dk, self.dv, self.dtables, self.dlens, msl, self.w.scale, ws,
                               partition_tokens=pt)
        return ws

    def oracle(self, seqs=None, threads=8):
        return oracle.decode_attention(self.q, self.k_pool, self.v_pool, self.ref_tables, self.lengths, self.w.scale,
                                       seqs=seqs, threads=threads)


def status_word(ws) -> int:
    return int(ws[:4].view(dtype=__import__("torch").int32).item())


def poison_unused_slots(k_pool: np.ndarray, v_pool: np.ndarray, tables: np.ndarray, lens: np.ndarray) -> int:
    """Fill every pool slot no sequence covers (free blocks, tails of partial blocks) with NaN, in place.

    Those slots may hold any bits in a real pool; a kernel must not let them reach an output
    (zero weight times NaN is NaN).  Returns the number of slots poisoned.
    """
    nb, _, bs, _ = k_pool.shape
    used = np.zeros((nb, bs), bool)
    for b, n in enumerate(lens):
        for t in range(int(n)):
            used[tables[b, t // bs], t % bs] = True
    nan = {np.dtype(np.uint16): np.uint16(0x7FC0), np.dtype(np.uint8): np.uint8(0x7F)}.get(k_pool.dtype, np.float32("nan"))
    for pool in (k_pool, v_pool):
        pool.transpose(0, 2, 1, 3)[~used] = nan
    return int((~used).sum())
