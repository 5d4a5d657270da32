"""GPU: FP8 (E4M3) pools -- append codes bit-exact against the oracle's encoder, decode within
the bf16 bound of the oracle's FP8 decode."""
import numpy as np
import pytest

import oracle
import synth
import synth.workloads as W
from gpu_cases import DecodeCase, check_close, poison_unused_slots, to_numpy, to_torch

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("in_dtype,scales", [("bf16", (1.0, 1.0)), ("bf16", (0.037, 2.5)), ("f32", (0.3, 0.011))])
def test_fp8_append_codes_are_bit_exact(in_dtype, scales):
    import torch
    import paged_kv_cache_280_gb300 as pa

    hkv, d, bs, nb, n = 4, 128, 16, 12, 37
    mags = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    edge = np.concatenate([mags, (mags[1:] + mags[:-1]) / 2, [500.0, 448.0, 464.0, 1e4, 2.0 ** -12, 0.0]])
    rng = np.random.default_rng(11)
    vals = np.concatenate([edge, -edge, rng.standard_normal(2 * n * hkv * d) * 4])[: 2 * n * hkv * d]
    rng.shuffle(vals)
    k = vals[: n * hkv * d].reshape(n, hkv, d) * scales[0]
    v = vals[n * hkv * d:].reshape(n, hkv, d) * scales[1]
    if in_dtype == "bf16":
        kn, vn = _bf16_bits(k), _bf16_bits(v)
    else:
        kn, vn = k.astype(np.float32), v.astype(np.float32)
    slots = synth.permutation(5, nb * bs)[:n].astype(np.int64)
    slots[3] = -1  # padding token: skipped
    kp = np.zeros((nb, hkv, bs, d), np.uint8)
    vp = np.zeros((nb, hkv, bs, d), np.uint8)
    dk = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device="cuda")
    dv = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache_fp8(to_torch(kn), to_torch(vn), dk, dv, to_torch(slots), *scales, status=status)
    oracle.reshape_and_cache_fp8(kn, vn, kp, vp, slots, *scales)
    assert np.array_equal(dk.cpu().numpy(), kp) and np.array_equal(dv.cpu().numpy(), vp)
    assert status.item() == 0


def _fp8_case(seed, hq, hkv, bs, lens=None, max_len=300):
    w = W.random_case(seed, 11 if lens is None else len(lens), hq, hkv, 128, bs, "bf16", max_len=max_len)
    c = DecodeCase(w, lengths=lens)
    ks, vs = 0.02 + 0.01 * (seed % 3), 0.05
    # FP8 pools: the oracle's codes of the bf16 pool values over the scales
    c.kq = oracle.e4m3_encode(oracle_bf16_values(c.k_pool) / np.float32(ks))
    c.vq = oracle.e4m3_encode(oracle_bf16_values(c.v_pool) / np.float32(vs))
    c.scales = (ks, vs)
    return c


def oracle_bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _run_fp8(c, partition_tokens=0):
    import torch
    import paged_kv_cache_280_gb300 as pa

    dq, dt, dl = to_torch(c.q), to_torch(c.tables), to_torch(c.lengths)
    dk, dv = torch.from_numpy(c.kq).cuda(), torch.from_numpy(c.vq).cuda()
    out = torch.empty_like(dq)
    n = pa.pa_decode_workspace_bytes(len(c.lengths), c.w.num_q_heads, c.w.num_kv_heads, 128)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    pa.pa_decode_attention_fp8(out, dq, dk, dv, *c.scales, dt, dl, int(c.lengths.max(initial=0)), c.w.scale, ws,
                               partition_tokens=partition_tokens)
    assert int(ws[:4].view(torch.int32).item()) == 0
    return to_numpy(out)


@pytest.mark.parametrize("hq,hkv,bs,pt", [(8, 8, 16, 0), (16, 8, 16, 0), (32, 8, 16, 0), (32, 4, 32, 0),
                                          (12, 4, 16, 0), (32, 8, 32, 64), (40, 8, 16, 0)])
def test_fp8_decode_matches_oracle(hq, hkv, bs, pt):
    lens = np.asarray(synth.uniform_ints(31 + hq, 11, 0, 300), np.int32)
    lens[:4] = [0, 1, bs, bs + 1]
    c = _fp8_case(300 + hq + bs, hq, hkv, bs, lens=lens)
    got = _run_fp8(c, pt)
    ref = oracle.decode_attention_fp8(c.q, c.kq, c.vq, *c.scales, c.ref_tables, c.lengths, c.w.scale, threads=8)
    check_close(got, ref, "bf16")
    assert np.array_equal(got[0], np.zeros_like(got[0]))  # empty sequence


def test_fp8_decode_ignores_nan_in_unused_slots():
    lens = np.asarray([5, 17, 33, 100, 1, 250], np.int32)
    c = _fp8_case(77, 32, 8, 16, lens=lens)
    poison_unused_slots(c.kq, c.vq, c.ref_tables, c.lengths)  # 0x7F: the NaN code
    assert np.sum(c.kq == 0x7F) > 0
    got = _run_fp8(c)
    ref = oracle.decode_attention_fp8(c.q, c.kq, c.vq, *c.scales, c.ref_tables, c.lengths, c.w.scale, threads=8)
    check_close(got, ref, "bf16")


@pytest.mark.parametrize("wl", ["long_context", "mha_b256"])
def test_fp8_full_size_workloads(wl):
    """The benchmark's FP8 configurations at full size, checked on sampled sequences: 4 x 131072
    tokens at 8 query heads per KV head with 2048-token partitions, and the 256-sequence MHA batch
    (one query head per KV head, the MMA's N padded)."""
    import torch
    import paged_kv_cache_280_gb300 as pa

    if wl == "long_context":
        w, pt = W.long_context(block_size=16), 2048
    else:
        w, pt = W.mha_b256_append(), 0
    c = DecodeCase(w)
    ks = vs = 1.0 / 64
    # Seeded codes spread over every finite E4M3 value (the NaN codes 0x7F and 0xFF left out):
    # inputs for both sides.  The oracle's encoder, a search over all codes per value, is too slow
    # for the pools' billion values, and the decode does not care where its codes came from.
    def codes(seed, shape):
        u = synth.uniform_ints(seed, int(np.prod(shape)), 0, 253)
        return np.where(u < 0x7F, u, u + 1).astype(np.uint8).reshape(shape)
    kq, vq = codes(280101, c.k_pool.shape), codes(280102, c.v_pool.shape)
    B = len(c.lengths)
    if wl == "long_context":
        sample = [0, 3]
    else:
        order = np.argsort(c.lengths)
        sample = sorted(set(order[:3].tolist() + order[-3:].tolist() + list(range(0, B, 41))))
    dq, dt, dl = to_torch(c.q), to_torch(c.tables), to_torch(c.lengths)
    dk, dv = torch.from_numpy(kq).cuda(), torch.from_numpy(vq).cuda()
    out = torch.empty_like(dq)
    ws = torch.zeros(pa.pa_decode_workspace_bytes(B, w.num_q_heads, w.num_kv_heads, 128), dtype=torch.uint8,
                     device="cuda")
    pa.pa_decode_attention_fp8(out, dq, dk, dv, ks, vs, dt, dl, int(c.lengths.max()), w.scale, ws, partition_tokens=pt)
    ref = oracle.decode_attention_fp8(c.q, kq, vq, ks, vs, c.ref_tables, c.lengths, w.scale, seqs=sample, threads=8)
    check_close(to_numpy(out), ref, "bf16", rows=sample)
    assert int(ws[:4].view(torch.int32).item()) == 0
