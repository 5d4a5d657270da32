"""GPU: prefix caching end to end.

Four requests share a 1024-token prefix (64 blocks) and differ in a 7-token
tail; 32/8 heads, d 128, bs 16.  Request 0 is prefilled in full and its
prefix registered; requests 1..3 reuse the 64 cached blocks and prefill only
their 7-token tails.  Their outputs must match the oracle over the full
context, and bit for bit the rows of an uncached full prefill of the same
prompt (the last query tile covers exactly the tail tokens either way).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_cases import check_close, to_numpy, to_torch
from oracle.alloc_model import RefAllocator

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS, PRE, TAIL, R = 32, 8, 128, 16, 1024, 7, 4


def test_cached_prefix_prefill():
    import torch
    import paged_kv_cache_280_gb300 as pa

    L = PRE + TAIL
    nb = 64 * 2 + 8 * R
    order = synth.permutation(synth.stream_seed(280108, 5), nb)
    lib, ref = pa.Allocator(nb, BS, free_order=order), RefAllocator(nb, BS, free_order=order.tolist())
    tokens = [[1000 + t for t in range(PRE)] + [r * 100 + t for t in range(TAIL)] for r in range(R)]
    kv = lambda tag, n: synth.normal(synth.stream_seed(280108, tag), n * HKV * D, "bf16").reshape(n, HKV, D)  # noqa: E731
    k_pre, v_pre = kv(1, PRE), kv(2, PRE)              # the shared prefix's K/V (same tokens, same KV)
    tails = [(kv(10 + r, TAIL), kv(20 + r, TAIL)) for r in range(R)]
    q = [synth.normal(synth.stream_seed(280108, 30 + r), L * HQ * D, "bf16").reshape(L, HQ, D) for r in range(R)]
    k_pool = synth.normal(synth.stream_seed(280108, 3), nb * HKV * BS * D, "bf16").reshape(nb, HKV, BS, D)
    v_pool = synth.normal(synth.stream_seed(280108, 4), nb * HKV * BS * D, "bf16").reshape(nb, HKV, BS, D)
    dk, dv = to_torch(k_pool), to_torch(v_pool)

    def write(slots, kk, vv):
        pa.pa_reshape_and_cache(to_torch(kk), to_torch(vv), dk, dv, to_torch(np.asarray(slots, np.int64)))
        oracle.reshape_and_cache(kk, vv, k_pool, v_pool, np.asarray(slots, np.int64))

    def prefill(seq, lens, chunk, qrows):
        tb, ln = lib.export_tables([seq], 80)
        rt = np.zeros_like(tb)
        rt[0, : len(ref.table(seq))] = ref.table(seq)
        assert np.array_equal(tb, rt) and ln.tolist() == [lens]
        out = torch.empty((chunk, HQ, D), dtype=torch.bfloat16, device="cuda")
        cu = np.array([0, chunk], np.int32)
        pa.pa_prefill_attention(out, to_torch(qrows), dk, dv, to_torch(tb), to_torch(ln), to_torch(cu), chunk,
                                1 / D ** 0.5)
        want = oracle.prefill_attention(qrows, k_pool, v_pool, rt, ln, cu, 1 / D ** 0.5)
        got = to_numpy(out)
        check_close(got, want, "bf16")
        return got

    # request 0: everything computed, then its prefix registered
    for a in (lib, ref):
        a.create(0)
        assert a.create_cached(90, tokens[0]) == 0  # nothing cached yet
        a.free_seq(90)
    s0, _ = lib.append(0, L)
    assert s0.tolist() == ref.append(0, L)[0]
    write(s0, np.concatenate([k_pre, tails[0][0]]), np.concatenate([v_pre, tails[0][1]]))
    prefill(0, L, L, q[0])
    lib.cache_prefix(0, tokens[0])
    ref.cache_prefix(0, tokens[0])
    assert lib.prefix_cache_stats() == ref.prefix_cache_stats() == {"cached_blocks": 64, "evictable_blocks": 0}
    for r in range(1, R):
        # cached: 1024 tokens reused, only the tail is appended and prefilled
        assert lib.create_cached(r, tokens[r]) == PRE and ref.create_cached(r, tokens[r]) == PRE
        assert lib.table(r) == lib.table(0)[:64]
        st, _ = lib.append(r, TAIL)
        assert st.tolist() == ref.append(r, TAIL)[0]
        write(st, *tails[r])
        got = prefill(r, L, TAIL, q[r][PRE:])
        # uncached: the same prompt in fresh blocks, prefilled in full
        sid = 100 + r
        for a in (lib, ref):
            a.create(sid)
        su, _ = lib.append(sid, L)
        assert su.tolist() == ref.append(sid, L)[0]
        write(su, np.concatenate([k_pre, tails[r][0]]), np.concatenate([v_pre, tails[r][1]]))
        full = prefill(sid, L, L, q[r])
        assert np.array_equal(got, full[PRE:])
        for a in (lib, ref):
            a.free_seq(sid)
    for r in range(R):
        assert lib.refcount(lib.table(0)[0]) == R
