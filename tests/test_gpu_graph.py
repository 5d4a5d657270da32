"""GPU: the decode step (append + decode) captured in a CUDA graph and replayed gives the same
output as eager launches, step after step, with new inputs written into the captured buffers."""
import numpy as np
import pytest

import synth.workloads as W
from gpu_cases import DecodeCase, to_numpy, to_torch

pytestmark = pytest.mark.gpu


def test_graph_replay_matches_eager():
    import torch
    import paged_kv_cache_280_gb300 as pa

    w = W.gqa4_b64(num_seqs=16, extra_tokens=8)
    c = DecodeCase(w)
    ids = list(range(16))
    max_blocks = c.max_blocks + 2
    B, Hq, Hkv, D = 16, w.num_q_heads, w.num_kv_heads, w.head_dim
    dk_e, dv_e = to_torch(c.k_pool), to_torch(c.v_pool)  # eager pools
    dk_g, dv_g = dk_e.clone(), dv_e.clone()               # graph pools
    lib_e = pa.Allocator(w.num_blocks, w.block_size, free_order=w.free_order())
    lib_g = pa.Allocator(w.num_blocks, w.block_size, free_order=w.free_order())
    for lib in (lib_e, lib_g):
        for s, n in enumerate(c.lengths):
            lib.create(s)
            lib.append(s, int(n))
    # captured buffers: inputs rewritten each step, outputs read each step
    g_q = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    g_kn = torch.empty((B, Hkv, D), dtype=torch.bfloat16, device="cuda")
    g_vn = torch.empty_like(g_kn)
    g_slots = torch.empty(B, dtype=torch.int64, device="cuda")
    g_tables = torch.empty((B, max_blocks), dtype=torch.int32, device="cuda")
    g_lens = torch.empty(B, dtype=torch.int32, device="cuda")
    g_out = torch.empty_like(g_q)
    n = pa.pa_decode_workspace_bytes(B, Hq, Hkv, D)
    ws_g = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ws_e = torch.zeros(n, dtype=torch.uint8, device="cuda")
    cap = max_blocks * w.block_size  # a length bound valid for every replay

    def step(dk, dv, q, kn, vn, slots, tables, lens, out, ws, max_len):
        pa.pa_reshape_and_cache(kn, vn, dk, dv, slots)
        pa.pa_decode_attention(out, q, dk, dv, tables, lens, max_len, w.scale, ws)

    # warm the library's per-kernel setup once, then capture
    s0, _ = lib_g.append_batch(ids)
    t0, l0 = lib_g.export_tables(ids, max_blocks)
    lib_e.append_batch(ids)
    for dst, src in ((g_slots, s0), (g_tables, t0), (g_lens, l0)):
        dst.copy_(torch.from_numpy(src))
    g_q.copy_(to_torch(w.queries(step=9)))
    g_kn.copy_(to_torch(w.new_tokens("k", B, step=9)))
    g_vn.copy_(to_torch(w.new_tokens("v", B, step=9)))
    step(dk_e, dv_e, g_q, g_kn, g_vn, g_slots, g_tables, g_lens, torch.empty_like(g_out), ws_e, cap)
    step(dk_g, dv_g, g_q, g_kn, g_vn, g_slots, g_tables, g_lens, g_out, ws_g, cap)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(dk_g, dv_g, g_q, g_kn, g_vn, g_slots, g_tables, g_lens, g_out, ws_g, cap)
    for k in range(3):
        # a new token per sequence: both allocators hand out the same slots and tables
        se, pe = lib_e.append_batch(ids)
        sg, pg = lib_g.append_batch(ids)
        assert se.tolist() == sg.tolist() and pe.size == pg.size == 0
        te, le = lib_e.export_tables(ids, max_blocks)
        q, kn, vn = w.queries(step=10 + k), w.new_tokens("k", B, step=10 + k), w.new_tokens("v", B, step=10 + k)
        out_e = torch.empty_like(g_out)
        step(dk_e, dv_e, to_torch(q), to_torch(kn), to_torch(vn), to_torch(se), to_torch(te), to_torch(le), out_e,
             ws_e, cap)
        for dst, src in ((g_q, q), (g_kn, kn), (g_vn, vn)):
            dst.copy_(to_torch(src))
        for dst, src in ((g_slots, sg), (g_tables, te), (g_lens, le)):
            dst.copy_(torch.from_numpy(src))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_numpy(g_out), to_numpy(out_e))
        assert torch.equal(dk_g, dk_e) and torch.equal(dv_g, dv_e)
    assert int(ws_g[:4].view(torch.int32).item()) == 0
