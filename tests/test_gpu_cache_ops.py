"""GPU: slot-mapped append and copy-on-write block copy are bit-exact against the oracle."""
import numpy as np
import pytest

import oracle
import synth
from gpu_cases import to_numpy, to_torch

pytestmark = pytest.mark.gpu


def _pools(seed, nb, hkv, bs, d, dtype):
    n = nb * hkv * bs * d
    k = synth.normal(synth.stream_seed(seed, 1), n, dtype).reshape(nb, hkv, bs, d)
    v = synth.normal(synth.stream_seed(seed, 2), n, dtype).reshape(nb, hkv, bs, d)
    return k, v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bs,d", [(16, 64), (16, 128), (32, 128), (32, 64)])
def test_reshape_and_cache_bitexact(dtype, bs, d):
    import torch
    import paged_kv_cache_280_gb300 as pa

    nb, hkv, n = 37, 3, 300
    k, v = _pools(7, nb, hkv, bs, d, dtype)
    kn = synth.normal(synth.stream_seed(7, 3), n * hkv * d, dtype).reshape(n, hkv, d)
    vn = synth.normal(synth.stream_seed(7, 4), n * hkv * d, dtype).reshape(n, hkv, d)
    slots = synth.permutation(11, nb * bs)[:n].astype(np.int64)
    slots[::17] = -1  # padding tokens are skipped
    dk, dv = to_torch(k), to_torch(v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(to_torch(kn), to_torch(vn), dk, dv, to_torch(slots), status=status)
    oracle.reshape_and_cache(kn, vn, k, v, slots)
    assert np.array_equal(to_numpy(dk), k) and np.array_equal(to_numpy(dv), v)
    assert status.item() == 0


def test_reshape_and_cache_flags_bad_slot_and_skips_it():
    import torch
    import paged_kv_cache_280_gb300 as pa

    nb, hkv, bs, d = 4, 2, 16, 64
    k, v = _pools(8, nb, hkv, bs, d, "bf16")
    kn = synth.normal(synth.stream_seed(8, 3), 3 * hkv * d, "bf16").reshape(3, hkv, d)
    slots = np.array([5, nb * bs, 9], np.int64)  # the middle slot is one past the pool
    dk, dv = to_torch(k), to_torch(v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(to_torch(kn), to_torch(kn), dk, dv, to_torch(slots), status=status)
    oracle.reshape_and_cache(kn[[0, 2]], kn[[0, 2]], k, v, slots[[0, 2]])
    assert np.array_equal(to_numpy(dk), k) and np.array_equal(to_numpy(dv), v)
    assert status.item() == pa.PA_DEV_BAD_SLOT


@pytest.mark.parametrize("dtype,bs,d,hkv", [("bf16", 16, 128, 8), ("f32", 32, 64, 4), ("bf16", 32, 128, 32)])
def test_copy_blocks_bitexact(dtype, bs, d, hkv):
    import torch
    import paged_kv_cache_280_gb300 as pa

    nb = 64
    k, v = _pools(9, nb, hkv, bs, d, dtype)
    perm = synth.permutation(12, nb)
    pairs = np.stack([perm[:20], perm[20:40]], 1).astype(np.int32)  # distinct, non-overlapping
    dk, dv = to_torch(k), to_torch(v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(dk, dv, to_torch(pairs), status=status)
    oracle.copy_blocks(k, v, pairs)
    assert np.array_equal(to_numpy(dk), k) and np.array_equal(to_numpy(dv), v)
    assert status.item() == 0


def test_copy_blocks_flags_bad_block():
    import torch
    import paged_kv_cache_280_gb300 as pa

    k, v = _pools(10, 8, 2, 16, 64, "f32")
    pairs = np.array([[1, 2], [3, 8], [4, 5]], np.int32)  # 8 is outside the pool
    dk, dv = to_torch(k), to_torch(v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(dk, dv, to_torch(pairs), status=status)
    oracle.copy_blocks(k, v, pairs[[0, 2]])
    assert np.array_equal(to_numpy(dk), k) and np.array_equal(to_numpy(dv), v)
    assert status.item() == pa.PA_DEV_BAD_BLOCK_ID


def test_host_checks_reject_bad_arguments():
    import torch
    import paged_kv_cache_280_gb300 as pa

    k = torch.zeros(4, 2, 16, 96, dtype=torch.bfloat16, device="cuda")  # head_dim 96 unsupported
    kn = torch.zeros(1, 2, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_reshape_and_cache(kn, kn, k, k, torch.zeros(1, dtype=torch.int64, device="cuda"))
    assert e.value.name == "PA_ERR_UNSUPPORTED"
    k = torch.zeros(4, 2, 24, 64, dtype=torch.float32, device="cuda")  # block 24 unsupported
    with pytest.raises(pa.PAError) as e:
        pa.pa_copy_blocks(k, k, torch.zeros(1, 2, dtype=torch.int32, device="cuda"))
    assert e.value.name == "PA_ERR_UNSUPPORTED"
