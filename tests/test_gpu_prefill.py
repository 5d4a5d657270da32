"""GPU parity of paged prefill (chunked causal) attention against the oracle.

Each case builds context lengths through the library allocator (tables
checked bit for bit against the reference allocator model), picks a chunk
per sequence -- empty, one token, a whole fresh prompt, or a tail of a
longer context -- and compares every output row with the fp64 oracle
within the bf16 bound |d| <= 1e-2 + 1e-2 |ref|.
"""
import numpy as np
import pytest

import oracle
import synth
import synth.workloads as W
from gpu_cases import DecodeCase, check_close, poison_unused_slots, to_numpy, to_torch, widen

pytestmark = pytest.mark.gpu


class PrefillCase:
    def __init__(self, seed, lengths, chunks, hq, hkv, d, bs):
        lengths = np.asarray(lengths, np.int32)
        demand = sum(-(-int(x) // bs) for x in lengths)
        w = W.random_case(seed, len(lengths), hq, hkv, d, bs, "bf16", max_len=1)
        w = W.scaled(w, lengths=lengths, num_blocks=int(demand * 1.25) + 4)
        self.c = DecodeCase(w)
        self.chunks = np.asarray(chunks, np.int32)
        self.cu = np.concatenate([[0], np.cumsum(self.chunks)]).astype(np.int32)
        T = int(self.cu[-1])
        self.q = synth.normal(synth.stream_seed(seed, 77), max(1, T) * hq * d, "bf16").reshape(max(1, T), hq, d)[:T]
        self.w = w

    def run(self, max_q_len=None, status=None):
        import torch
        import paged_kv_cache_280_gb300 as pa

        c = self.c.device()
        self.dq = to_torch(self.q) if len(self.q) else torch.empty((0,) + self.q.shape[1:], dtype=torch.bfloat16,
                                                                      device="cuda")
        self.dout = torch.full_like(self.dq, float("nan")) if len(self.q) else self.dq
        mq = int(self.chunks.max(initial=0)) if max_q_len is None else max_q_len
        if len(self.q):
            pa.pa_prefill_attention(self.dout, self.dq, c.dk, c.dv, c.dtables, c.dlens, to_torch(self.cu), mq,
                                    self.w.scale, status=status)
        return to_numpy(self.dout)

    def oracle(self, seqs=None):
        return oracle.prefill_attention(self.q, self.c.k_pool, self.c.v_pool, self.c.ref_tables, self.c.lengths,
                                        self.cu, self.w.scale, seqs=seqs, threads=8)


@pytest.mark.parametrize("hq,hkv,d,bs", [(8, 8, 64, 16), (32, 8, 128, 16), (16, 2, 128, 32), (12, 4, 64, 32),
                                         (8, 1, 128, 16), (6, 2, 64, 16)])
def test_prefill_ragged_batch(hq, hkv, d, bs):
    # empty chunk, one token, a fresh prompt, chunk tails of longer contexts, several query tiles
    lengths = [37, 1, 130, 64, 200, 90, 17]
    chunks = [0, 1, 130, 20, 150, 9, 17]
    case = PrefillCase(280100 + hq + d + bs, lengths, chunks, hq, hkv, d, bs)
    got = case.run()
    check_close(got, case.oracle(), "bf16")


def test_prefill_parallel_sampling_prompts():
    """Prompt prefill of the parallel-sampling workload's shape: 1031-token fresh prompts, 32/8 heads, d 128."""
    case = PrefillCase(280104, [1031] * 4, [1031] * 4, 32, 8, 128, 16)
    got = case.run()
    check_close(got, case.oracle(), "bf16")


def test_prefill_grid_larger_than_chunks_and_bad_chunk():
    """max_q_len above every chunk only adds idle CTAs; a chunk longer than its context is flagged and skipped."""
    import torch
    import paged_kv_cache_280_gb300 as pa

    case = PrefillCase(280105, [40, 10, 70], [12, 11, 70], 16, 4, 128, 16)  # sequence 1: 11 queries, 10 keys
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = case.run(max_q_len=300, status=status)
    assert status.item() & 0x4  # PA_DEV_BAD_SEQ_LEN
    rows = list(range(0, 12)) + list(range(23, 93))
    ref = oracle.prefill_attention(case.q, case.c.k_pool, case.c.v_pool, case.c.ref_tables, case.c.lengths,
                                   case.cu, case.w.scale, seqs=[0, 2])
    check_close(got, ref, "bf16", rows=rows)
    assert np.all(np.isnan(widen(got[12:23])))  # the flagged sequence's rows are left untouched


def test_one_token_chunks_match_decode():
    """A one-token chunk per sequence is decode: the prefill kernel and the decode kernel agree with the oracle."""
    import paged_kv_cache_280_gb300 as pa

    lengths = [1, 16, 17, 250, 33]
    case = PrefillCase(280106, lengths, [1] * 5, 32, 8, 128, 16)
    got = case.run()
    ref = oracle.decode_attention(case.q, case.c.k_pool, case.c.v_pool, case.c.ref_tables, case.c.lengths,
                                  case.w.scale)
    check_close(got, ref, "bf16")


@pytest.mark.parametrize("bs", [16, 32])
def test_prefill_ignores_nan_in_unused_slots(bs):
    """Free blocks and the unfilled tail of each last block hold NaN; no output may see them."""
    lengths = [37, 130, 17, 64, 91]
    chunks = [5, 130, 17, 64, 3]  # tiles that end mid-context, at odd block counts, and at the end
    case = PrefillCase(280107 + bs, lengths, chunks, 32, 8, 128, bs)
    assert poison_unused_slots(case.c.k_pool, case.c.v_pool, case.c.ref_tables, case.c.lengths) > 0
    got = case.run()
    check_close(got, case.oracle(), "bf16")


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (32, 8, 32), (16, 2, 16)])
def test_prefill_nan_tail_read_by_an_earlier_unit(hq, hkv, bs):
    """A unit that ends a few tokens before its chunk's end can still load the sequence's partial
    last block (the NaN slots past the context's end): its output must not see them."""
    lengths = [106, 116, 200]
    chunks = [69, 69, 133]  # each chunk's last unit holds 5 tokens, so the unit before ends 5 keys short
    case = PrefillCase(280110 + hq + bs, lengths, chunks, hq, hkv, 128, bs)
    assert poison_unused_slots(case.c.k_pool, case.c.v_pool, case.c.ref_tables, case.c.lengths) > 0
    got = case.run()
    check_close(got, case.oracle(), "bf16")
