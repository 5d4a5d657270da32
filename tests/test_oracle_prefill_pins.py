"""Pins of the oracle's paged prefill (chunked causal) attention.

Each pin ties the oracle to something other than itself:
  * a one-token chunk is decode attention at the same length (the oracle's
    decode path, itself pinned by test_oracle_pins.py);
  * brute force in matrix form on never-paged contiguous tensors:
    softmax(scale Q K^T + causal mask) V, with the mask written as a
    position comparison over the whole sequence;
  * the first token of a fresh sequence sees only itself, so its output is
    exactly V[0];
  * invariance under any relabelling of the physical blocks;
  * splitting a chunk in two (the second call seeing the first one's tokens
    as context) changes no output row.
"""
import math

import numpy as np
import pytest

import oracle


def _bf16(x):
    """fp32 -> bf16 bit patterns (round to nearest even), and the values they hold."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r, (r.astype(np.uint32) << 16).view(np.float32)


def _case(seed, lens, chunks, hq, hkv, d, bs, extra_blocks=3):
    """Contiguous K/V per sequence, scattered into a pool by a seeded permutation."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    nblk = [-(-L // bs) for L in lens]
    nb = sum(nblk) + extra_blocks
    perm = rng.permutation(nb)
    maxb = max(1, max(nblk))
    tables = np.zeros((B, maxb), np.int32)
    kp_f = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    vp_f = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    kc, vc, pos = [], [], 0
    for b, L in enumerate(lens):
        tables[b, : nblk[b]] = perm[pos: pos + nblk[b]]
        pos += nblk[b]
        kc.append(rng.standard_normal((L, hkv, d)).astype(np.float32))
        vc.append(rng.standard_normal((L, hkv, d)).astype(np.float32))
        for t in range(L):
            kp_f[tables[b, t // bs], :, t % bs] = kc[b][t]
            vp_f[tables[b, t // bs], :, t % bs] = vc[b][t]
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = rng.standard_normal((int(cu[-1]), hq, d)).astype(np.float32)
    return q, kp_f, vp_f, tables, np.asarray(lens, np.int32), cu, kc, vc


def _brute(q, kc, vc, lens, cu, hq, hkv, scale):
    """softmax(scale Q K^T + mask) V per sequence and head, on the contiguous tensors."""
    G = hq // hkv
    out = np.zeros(q.shape, np.float64)
    for b, L in enumerate(lens):
        n = cu[b + 1] - cu[b]
        if n == 0:
            continue
        Q = q[cu[b]:cu[b + 1]].astype(np.float64)  # [n][hq][d]
        qpos = np.arange(L - n, L)[:, None]
        kpos = np.arange(L)[None, :]
        mask = np.where(kpos <= qpos, 0.0, -np.inf)
        for h in range(hq):
            K = kc[b][:, h // G].astype(np.float64)
            V = vc[b][:, h // G].astype(np.float64)
            S = scale * Q[:, h] @ K.T + mask
            P = np.exp(S - S.max(axis=1, keepdims=True))
            out[cu[b]:cu[b + 1], h] = (P / P.sum(axis=1, keepdims=True)) @ V
    return out


@pytest.mark.parametrize("hq,hkv,d,bs", [(4, 4, 16, 4), (8, 2, 32, 16), (6, 3, 8, 32)])
def test_prefill_matches_brute_force(hq, hkv, d, bs):
    lens, chunks = [7, 40, 33, 1, 0, 19], [7, 12, 33, 1, 0, 5]
    q, kp, vp, tables, lens_a, cu, kc, vc = _case(11 + hq, lens, chunks, hq, hkv, d, bs)
    scale = 1.0 / math.sqrt(d)
    got = oracle.prefill_attention(q, kp, vp, tables, lens_a, cu, scale)
    want = _brute(q, kc, vc, lens_a, cu, hq, hkv, scale)
    assert np.max(np.abs(got - want)) < 1e-12


def test_prefill_bf16_widening_matches_brute_force():
    lens, chunks = [20, 9], [20, 4]
    q, kp, vp, tables, lens_a, cu, kc, vc = _case(5, lens, chunks, 8, 2, 16, 16)
    qb, qv = _bf16(q)
    kb, kv = _bf16(kp)
    vb, vv = _bf16(vp)
    got = oracle.prefill_attention(qb, kb, vb, tables, lens_a, cu, 0.25)
    kcv = [np.stack([kv[tables[b, t // 16], :, t % 16] for t in range(L)]) for b, L in enumerate(lens)]
    vcv = [np.stack([vv[tables[b, t // 16], :, t % 16] for t in range(L)]) for b, L in enumerate(lens)]
    want = _brute(qv, kcv, vcv, lens_a, cu, 8, 2, 0.25)
    assert np.max(np.abs(got - want)) < 1e-12


def test_one_token_chunk_is_decode():
    lens = [1, 16, 17, 50, 3]
    q, kp, vp, tables, lens_a, cu, _, _ = _case(3, lens, [1] * len(lens), 8, 4, 16, 16)
    pre = oracle.prefill_attention(q, kp, vp, tables, lens_a, cu, 0.3)
    dec = oracle.decode_attention(q, kp, vp, tables, lens_a, 0.3)
    assert np.max(np.abs(pre - dec)) < 1e-13


def test_first_token_of_fresh_sequence_is_its_value():
    q, kp, vp, tables, lens_a, cu, kc, vc = _case(9, [24], [24], 4, 2, 8, 16)
    out = oracle.prefill_attention(q, kp, vp, tables, lens_a, cu, 0.7)
    for h in range(4):
        assert np.array_equal(out[0, h], vc[0][0, h // 2].astype(np.float64))


def test_physical_relabelling_changes_nothing():
    q, kp, vp, tables, lens_a, cu, _, _ = _case(21, [30, 45], [10, 45], 4, 4, 16, 16)
    base = oracle.prefill_attention(q, kp, vp, tables, lens_a, cu, 0.25)
    perm = np.random.default_rng(4).permutation(kp.shape[0])
    inv = np.argsort(perm)
    kp2, vp2 = kp[inv], vp[inv]  # block b moves to perm[b]
    t2 = perm[tables].astype(np.int32)
    assert np.array_equal(oracle.prefill_attention(q, kp2, vp2, t2, lens_a, cu, 0.25), base)


def test_chunk_split_changes_no_row():
    L, n, n1 = 57, 40, 13
    q, kp, vp, tables, lens_a, cu, _, _ = _case(8, [L], [n], 4, 2, 16, 16)
    whole = oracle.prefill_attention(q, kp, vp, tables, lens_a, cu, 0.2)
    first = oracle.prefill_attention(q[:n1], kp, vp, tables, np.array([L - n + n1], np.int32),
                                     np.array([0, n1], np.int32), 0.2)
    second = oracle.prefill_attention(q[n1:], kp, vp, tables, lens_a, np.array([0, n - n1], np.int32), 0.2)
    assert np.array_equal(np.concatenate([first, second]), whole)


def test_bad_chunk_is_refused():
    q, kp, vp, tables, lens_a, cu, _, _ = _case(1, [5], [5], 2, 2, 8, 16)
    with pytest.raises(oracle.OracleError):
        oracle.prefill_attention(np.zeros((6, 2, 8), np.float32), kp, vp, tables, lens_a,
                                 np.array([0, 6], np.int32), 0.5)
