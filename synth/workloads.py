"""Workload recipes: shapes, sizes and which seeded stream feeds which input.

The recipes follow the workloads of the PagedAttention pages: 16-token
blocks scattered through a physical pool (a seeded Fisher-Yates order of
the free list), the skewed request-length mix of the waste simulation on
the ohmygp.com page, refcount-shared prompt prefixes for parallel sampling,
and 128K-token contexts (8192-entry block tables, page 1 follow-up 1).
Nothing here computes attention, slots or copies: the allocator and the
kernels (or the oracle) do that from these inputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

import synth

# stream tags (kept apart by synth.stream_seed)
TAG_LENGTHS = 1
TAG_Q = 2
TAG_K_POOL = 3
TAG_V_POOL = 4
TAG_FREE_ORDER = 5
TAG_TAILS = 6
TAG_K_NEW = 7
TAG_V_NEW = 8
TAG_PROMPT_K = 9
TAG_PROMPT_V = 10


def step_tag(tag: int, step: int) -> int:
    """Tag of a per-decode-step stream (new tokens, queries of step ``step``)."""
    return 1000 + 64 * step + tag


@dataclass
class Workload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str  # "f32" or "bf16"
    lengths: np.ndarray  # context length of each sequence before the step's append
    num_blocks: int
    scale: float
    append_one: bool = False  # the decode step appends one new token per sequence first
    partition_tokens: int = 0  # 0 = automatic split
    # parallel sampling with copy-on-write
    prompts: int = 0
    samples: int = 0
    prompt_len: int = 0
    tail_max: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        if self.prompts:
            return self.prompts * self.samples
        return int(len(self.lengths))

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def stream(self, tag: int) -> int:
        return synth.stream_seed(self.seed, tag)

    def free_order(self) -> np.ndarray:
        """Initial free-list order of the block pool (seeded permutation)."""
        return synth.permutation(self.stream(TAG_FREE_ORDER), self.num_blocks)

    def pool_shape(self):
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def pool_values(self, which: str) -> np.ndarray:
        """Initial contents of the K or V pool (every slot, used or not)."""
        tag = TAG_K_POOL if which == "k" else TAG_V_POOL
        n = int(np.prod(self.pool_shape()))
        return synth.normal(self.stream(tag), n, self.dtype).reshape(self.pool_shape())

    def queries(self, step: int = 0) -> np.ndarray:
        n = self.num_seqs * self.num_q_heads * self.head_dim
        tag = TAG_Q if step == 0 else step_tag(TAG_Q, step)
        return synth.normal(self.stream(tag), n, self.dtype).reshape(
            self.num_seqs, self.num_q_heads, self.head_dim
        )

    def new_tokens(self, which: str, n_tokens: int, step: int = 0) -> np.ndarray:
        tag = step_tag(TAG_K_NEW if which == "k" else TAG_V_NEW, step)
        n = n_tokens * self.num_kv_heads * self.head_dim
        return synth.normal(self.stream(tag), n, self.dtype).reshape(
            n_tokens, self.num_kv_heads, self.head_dim
        )

    def prompt_tokens(self, which: str) -> np.ndarray:
        tag = TAG_PROMPT_K if which == "k" else TAG_PROMPT_V
        n = self.prompts * self.prompt_len * self.num_kv_heads * self.head_dim
        return synth.normal(self.stream(tag), n, self.dtype).reshape(
            self.prompts * self.prompt_len, self.num_kv_heads, self.head_dim
        )

    def tails(self) -> np.ndarray:
        """Per-sample divergent tail lengths U[0, tail_max], prompt-major order."""
        return synth.uniform_ints(self.stream(TAG_TAILS), self.prompts * self.samples, 0, self.tail_max)

    def kv_token_bytes(self) -> int:
        """Bytes of K plus V for one token position across all KV heads."""
        return 2 * self.num_kv_heads * self.head_dim * self.elem_bytes


def _blocks(lengths, bs) -> int:
    return int(sum((int(x) + bs - 1) // bs for x in lengths))


def tiny_fp32() -> Workload:
    """4 sequences {5,17,33,48}, MHA 4 heads, d 64, fp32, pool of 32 blocks."""
    return Workload(
        name="tiny_fp32_b4_mha4_d64_bs16",
        seed=280001,
        num_q_heads=4,
        num_kv_heads=4,
        head_dim=64,
        block_size=16,
        dtype="f32",
        lengths=np.array([5, 17, 33, 48], np.int32),
        num_blocks=32,
        scale=1.0 / math.sqrt(64.0),
    )


def gqa4_b64(num_seqs: int = 64, extra_tokens: int = 0) -> Workload:
    """bf16 decode batch of 64 skew-mixed lengths, 32 query / 8 KV heads, d 128.

    ``extra_tokens`` reserves pool room for that many later appends per
    sequence (decode steps); the pool is total demand + 10 %.
    """
    seed = 280002
    lengths = synth.lengths_mix(synth.stream_seed(seed, TAG_LENGTHS), num_seqs)
    demand = _blocks(lengths + extra_tokens, 16)
    return Workload(
        name=f"gqa4_b{num_seqs}_hq32_hkv8_d128_bs16_bf16",
        seed=seed,
        num_q_heads=32,
        num_kv_heads=8,
        head_dim=128,
        block_size=16,
        dtype="bf16",
        lengths=lengths,
        num_blocks=int(math.ceil(1.1 * demand)),
        scale=1.0 / math.sqrt(128.0),
        extra={"extra_tokens": extra_tokens},
    )


def mha_b256_append(num_seqs: int = 256) -> Workload:
    """bf16 batch of 256 skew-mixed lengths, MHA 32 heads, d 128; append one token, then decode."""
    seed = 280003
    lengths = synth.lengths_mix(synth.stream_seed(seed, TAG_LENGTHS), num_seqs)
    demand = _blocks(lengths + 1, 16)
    return Workload(
        name=f"mha_b{num_seqs}_h32_d128_bs16_bf16_append1",
        seed=seed,
        num_q_heads=32,
        num_kv_heads=32,
        head_dim=128,
        block_size=16,
        dtype="bf16",
        lengths=lengths,
        num_blocks=int(math.ceil(1.1 * demand)),
        scale=1.0 / math.sqrt(128.0),
        append_one=True,
    )


def cow_sampling(prompts: int = 16, samples: int = 8, prompt_len: int = 1031, tail_max: int = 256) -> Workload:
    """Parallel sampling: prompts of 1024 + 7 tokens shared by 8 samples each, tails U[0,256]."""
    seed = 280004
    bs = 16
    per_sample = (prompt_len % bs + tail_max + bs - 1) // bs + 1
    demand = prompts * ((prompt_len + bs - 1) // bs) + prompts * samples * per_sample
    return Workload(
        name=f"cow_p{prompts}x{samples}_len{prompt_len}_tail{tail_max}_hq32_hkv8_d128_bs16_bf16",
        seed=seed,
        num_q_heads=32,
        num_kv_heads=8,
        head_dim=128,
        block_size=bs,
        dtype="bf16",
        lengths=np.zeros(0, np.int32),
        num_blocks=int(math.ceil(1.1 * demand)),
        scale=1.0 / math.sqrt(128.0),
        prompts=prompts,
        samples=samples,
        prompt_len=prompt_len,
        tail_max=tail_max,
    )


def long_context(block_size: int = 16, num_seqs: int = 4, seq_len: int = 131072, partition_tokens: int = 2048) -> Workload:
    """4 x 128K-token contexts, 64 query / 8 KV heads, d 128, bf16, split into 2048-token partitions."""
    seed = 280005
    lengths = np.full(num_seqs, seq_len, np.int32)
    return Workload(
        name=f"long_b{num_seqs}x{seq_len}_hq64_hkv8_d128_bs{block_size}_bf16_p{partition_tokens}",
        seed=seed,
        num_q_heads=64,
        num_kv_heads=8,
        head_dim=128,
        block_size=block_size,
        dtype="bf16",
        lengths=lengths,
        num_blocks=int(math.ceil(1.1 * _blocks(lengths, block_size))),
        scale=1.0 / math.sqrt(128.0),
        partition_tokens=partition_tokens,
    )


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with fields replaced (smaller parity cases of the same recipe)."""
    return replace(w, **changes)


def random_case(seed: int, num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                block_size: int, dtype: str, max_len: int, min_len: int = 0, slack: float = 1.25) -> Workload:
    """A small ragged case with uniform lengths in [min_len, max_len]."""
    lengths = synth.uniform_ints(synth.stream_seed(seed, TAG_LENGTHS), num_seqs, min_len, max_len)
    demand = max(1, _blocks(lengths + 1, block_size))
    return Workload(
        name=f"rand{seed}_b{num_seqs}_hq{num_q_heads}_hkv{num_kv_heads}_d{head_dim}_bs{block_size}_{dtype}",
        seed=seed,
        num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        block_size=block_size,
        dtype=dtype,
        lengths=lengths,
        num_blocks=int(math.ceil(slack * demand)) + 1,
        scale=1.0 / math.sqrt(float(head_dim)),
    )
