"""Pins of the attention oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle -- a wrong block
or slot index, a transposed head mapping, a dropped scale, a missing
max-subtraction term, a wrong reduce weight -- fails at least one of them:

* a hand-derived two-token closed form (golden fixture);
* a library routine on never-paged contiguous tensors (scipy's softmax and
  numpy matmul), with the same data paged into a scattered pool;
* invariance under any permutation of physical block ids (bit-identical);
* closed forms: one token -> that V row exactly; q = 0 or all keys equal ->
  the mean of V; one dominant score -> that V row; empty sequence -> 0;
* GQA equals MHA with duplicated KV heads (bit-identical);
* the split-sequence reduce equals the unsplit result (1e-12).
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth
from golden_io import table


def _page(K, V, bs, num_blocks, order, Hkv=1):
    """Scatter contiguous per-sequence K/V ([B][Hkv][len][D]) into a pool following `order`."""
    B = len(K)
    D = K[0].shape[-1]
    kp = np.full((num_blocks, Hkv, bs, D), 7.0, np.float32)
    vp = np.full((num_blocks, Hkv, bs, D), -7.0, np.float32)
    maxb = max(1, max(-(-k.shape[1] // bs) for k in K))
    bt = np.zeros((B, maxb), np.int32)
    it = iter(order)
    for b in range(B):
        n = K[b].shape[1]
        for j in range(-(-n // bs)):
            phys = next(it)
            bt[b, j] = phys
            t0, t1 = j * bs, min(n, (j + 1) * bs)
            kp[phys, :, : t1 - t0] = K[b][:, t0:t1]
            vp[phys, :, : t1 - t0] = V[b][:, t0:t1]
    return kp, vp, bt


def _rand_case(seed, lens, Hq, Hkv, D, bs):
    s = synth.stream_seed(seed, 1)
    K = [synth.normal(s, Hkv * n * D, "f32", offset=10_000_000 * b).reshape(Hkv, n, D) for b, n in enumerate(lens)]
    s = synth.stream_seed(seed, 2)
    V = [synth.normal(s, Hkv * n * D, "f32", offset=10_000_000 * b).reshape(Hkv, n, D) for b, n in enumerate(lens)]
    q = synth.normal(synth.stream_seed(seed, 3), len(lens) * Hq * D, "f32").reshape(len(lens), Hq, D)
    return q, K, V


def test_two_token_closed_form():
    g, _ = table("two_token_attention.txt")
    D = int(g["D"][0])
    nb = int(g["num_blocks"][0])
    phys = int(g["physical_block"][0])
    kp = np.full((nb, 1, 16, D), 9.0, np.float32)
    vp = np.full((nb, 1, 16, D), 9.0, np.float32)
    kp[phys, 0, 0], kp[phys, 0, 1] = [float(x) for x in g["k_t0"]], [float(x) for x in g["k_t1"]]
    vp[phys, 0, 0], vp[phys, 0, 1] = [float(x) for x in g["v_t0"]], [float(x) for x in g["v_t1"]]
    q = np.array([[[float(x) for x in g["q0"]], [float(x) for x in g["q1"]]]], np.float32)
    bt = np.array([[phys]], np.int32)
    out = oracle.decode_attention(q, kp, vp, bt, np.array([2], np.int32), float(g["scale"][0]))
    want = np.array([[float(x) for x in g["out0"]], [float(x) for x in g["out1"]]])
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("bs", [16, 32])
def test_matches_library_softmax_on_contiguous(bs):
    lens = [1, 15, 16, 17, 40, 75]
    Hq = Hkv = 2
    D = 64
    q, K, V = _rand_case(1, lens, Hq, Hkv, D, bs)
    nb = 40
    kp, vp, bt = _page(K, V, bs, nb, synth.permutation(17, nb), Hkv)
    scale = 1 / math.sqrt(D)
    out = oracle.decode_attention(q, kp, vp, bt, np.array(lens, np.int32), scale)
    for b, n in enumerate(lens):
        for h in range(Hq):
            Kc = K[b][h].astype(np.float64)
            Vc = V[b][h].astype(np.float64)
            w = softmax(scale * (Kc @ q[b, h].astype(np.float64)))
            np.testing.assert_allclose(out[b, h], w @ Vc, rtol=0, atol=1e-12)


def test_physical_permutation_invariance_bitexact():
    lens = [3, 16, 33, 70, 128]
    q, K, V = _rand_case(2, lens, 4, 2, 64, 16)
    outs = []
    for perm_seed in (1, 2, 3):
        kp, vp, bt = _page(K, V, 16, 64, synth.permutation(perm_seed, 64), 2)
        outs.append(oracle.decode_attention(q, kp, vp, bt, np.array(lens, np.int32), 0.125))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_closed_forms():
    D, bs = 64, 16
    rng_q, K, V = _rand_case(3, [1, 20, 20, 20], 1, 1, D, bs)
    K[2][:] = K[2][:, :1]  # all keys equal
    K[3][0, 7] *= 0.0
    K[3][0, 7] += 1000.0 * np.sign(rng_q[3, 0])  # one dominant key (score ~ 1000*|q|_1*scale)
    q = rng_q.copy()
    q[1] = 0.0  # zero query
    kp, vp, bt = _page(K, V, bs, 16, synth.permutation(5, 16), 1)
    lens = np.array([1, 20, 20, 20], np.int32)
    out = oracle.decode_attention(q, kp, vp, bt, lens, 1 / 8)
    assert np.array_equal(out[0, 0], V[0][0, 0].astype(np.float64))  # one token: exactly V
    np.testing.assert_allclose(out[1, 0], V[1][0].astype(np.float64).mean(0), atol=1e-14)
    np.testing.assert_allclose(out[2, 0], V[2][0].astype(np.float64).mean(0), atol=1e-14)
    np.testing.assert_allclose(out[3, 0], V[3][0, 7].astype(np.float64), atol=1e-12)


def test_empty_sequence_gives_zero():
    q, K, V = _rand_case(4, [5], 2, 1, 64, 16)
    kp, vp, bt = _page(K, V, 16, 4, [2, 0, 1, 3], 1)
    out = oracle.decode_attention(q, kp, vp, bt, np.array([0], np.int32), 0.1)
    assert np.array_equal(out, np.zeros_like(out))


def test_gqa_equals_mha_with_duplicated_kv_heads():
    lens = [9, 31, 64]
    Hq, Hkv, D = 8, 2, 64
    q, K, V = _rand_case(6, lens, Hq, Hkv, D, 16)
    kp, vp, bt = _page(K, V, 16, 24, synth.permutation(8, 24), Hkv)
    gqa = oracle.decode_attention(q, kp, vp, bt, np.array(lens, np.int32), 0.125)
    G = Hq // Hkv
    K2 = [np.repeat(k, G, axis=0) for k in K]  # kv head h of the MHA copy = original h // G
    V2 = [np.repeat(v, G, axis=0) for v in V]
    kp2, vp2, bt2 = _page(K2, V2, 16, 24, synth.permutation(8, 24), Hq)
    mha = oracle.decode_attention(q, kp2, vp2, bt2, np.array(lens, np.int32), 0.125)
    assert np.array_equal(gqa, mha)


def test_bf16_inputs_widen_exactly():
    lens = [10, 21]
    q, K, V = _rand_case(7, lens, 2, 1, 64, 16)

    def to_bf16_bits(a):
        u = a.astype(np.float32).view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    def from_bits(b):
        return (b.astype(np.uint32) << 16).view(np.float32)

    kp, vp, bt = _page(K, V, 16, 8, list(range(8)), 1)
    qb, kb, vb = to_bf16_bits(q), to_bf16_bits(kp), to_bf16_bits(vp)
    out_bits = oracle.decode_attention(qb, kb, vb, bt, np.array(lens, np.int32), 0.125)
    out_f32 = oracle.decode_attention(from_bits(qb), from_bits(kb), from_bits(vb), bt, np.array(lens, np.int32), 0.125)
    assert np.array_equal(out_bits, out_f32)


@pytest.mark.parametrize("P", [16, 32, 48, 2048])
def test_split_reduce_equals_unsplit(P):
    lens = [0, 1, 16, 47, 100, 257]
    q, K, V = _rand_case(9, lens, 4, 2, 64, 16)
    kp, vp, bt = _page(K, V, 16, 48, synth.permutation(10, 48), 2)
    L = np.array(lens, np.int32)
    full = oracle.decode_attention(q, kp, vp, bt, L, 0.2)
    m, l, o = oracle.decode_partials(q, kp, vp, bt, L, 0.2, P)
    comb = oracle.combine_partials(m, l, o)
    np.testing.assert_allclose(comb, full, rtol=0, atol=1e-12)
    # each partition's (m, l) is its own max and sum: the first partition of a
    # long sequence can be checked against a library softmax normaliser
    b = 5
    s = 0.2 * (K[b][0, :P].astype(np.float64) @ q[b, 0].astype(np.float64))
    assert m[b, 0, 0] == pytest.approx(s.max(), abs=1e-12)
    assert l[b, 0, 0] == pytest.approx(np.exp(s - s.max()).sum(), rel=1e-13)


def test_bad_block_id_is_reported():
    q, K, V = _rand_case(11, [20], 1, 1, 64, 16)
    kp, vp, bt = _page(K, V, 16, 4, [0, 1, 2, 3], 1)
    bt[0, 1] = 4  # outside the 4-block pool
    with pytest.raises(oracle.OracleError):
        oracle.decode_attention(q, kp, vp, bt, np.array([20], np.int32), 0.1)
