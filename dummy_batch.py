"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the method: it only draws token ids, masks
and Gaussian Q/K/V/dO tensors from a seed, in the shapes of the workloads below.
Both sides of every parity check (the CUDA library and the CPU oracle) receive
the same arrays from here.

The batch follows the parameters of ``create_dummy_batch(batch_size,
num_unique_prompts, prompt_len, response_len)`` named on "Performance
Benchmarks" (section "Usage Tips for Optimal Performance"); that page gives no
value distribution or row order, so ids are uniform over the vocabulary, the
rows of a group are scattered by a seeded permutation, and response lengths,
when they vary, are uniform over the stated range with right padding.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    G: int            # unique prompts
    n: int            # responses per prompt
    P: int            # prompt length
    R: int            # padded response width
    vocab: int
    Hq: int
    Hkv: int
    D: int
    dtype: str        # "bf16" or "f32"
    backward: bool
    resp_len_range: tuple | None = None   # (lo, hi) inclusive, right padded
    hidden: int = 0   # width of an extra [B, L, hidden] tensor to pack

    @property
    def B(self) -> int:
        return self.G * self.n

    @property
    def L(self) -> int:
        return self.P + self.R


WORKLOADS = {
    # 2 unique prompts x 2 responses, prompt 128, response 32, 2 Q / 1 KV heads,
    # head_dim 64, fp32, forward + backward
    "tiny": Workload("tiny", 2, 2, 128, 32, 32000, 2, 1, 64, "f32", True),
    # Qwen3-0.6B attention shape, 2 unique prompts x 8 responses, 8192 + 512,
    # forward only
    "qwen3_0p6b": Workload("qwen3_0p6b", 2, 8, 8192, 512, 151936, 16, 8, 128, "bf16", False),
    # the worked redundancy example: one 10240-token prompt x 10 responses of
    # 1024 tokens, forward + backward
    "worked_example": Workload("worked_example", 1, 10, 10240, 1024, 151936, 16, 8, 128,
                               "bf16", True),
    # long context: 4 prompts of 32768 x 8 responses of 2048
    "long_context": Workload("long_context", 4, 8, 32768, 2048, 151936, 16, 8, 128, "bf16", True),
    # full pipeline: 8 prompts x 8, prompt 4096, responses 256..1024 right
    # padded to 1024, hidden 1024 packed and reconstructed
    "pipeline": Workload("pipeline", 8, 8, 4096, 1024, 151936, 16, 8, 128, "bf16", True,
                         resp_len_range=(256, 1024), hidden=1024),
    # the same with 64 distinct prompts (nothing to deduplicate)
    "pipeline_nodedup": Workload("pipeline_nodedup", 64, 1, 4096, 1024, 151936, 16, 8, 128,
                                 "bf16", True, resp_len_range=(256, 1024), hidden=1024),
    # one group of the long-context workload (1 prompt of 32768 x 8 responses
    # of 2048): the same kernels and tiles on a quarter of the data, the size
    # used for single-kernel profiler captures
    "long_context_1g": Workload("long_context_1g", 1, 8, 32768, 2048, 151936, 16, 8, 128, "bf16", True),
}

SEED_BASE = 1000


def make_batch(G, n, P, R, vocab, seed, shuffle=True, resp_len_range=None,
               pad_id=0, prompt_pad_range=None):
    """Draw ``input_ids [B, L]`` (int64), ``attention_mask [B, L]`` (uint8 or
    None) and ``position_ids [B, L]`` (int64).

    G prompts of P uniform ids each; every row is one of them followed by R
    uniform response ids.  ``resp_len_range=(lo, hi)`` right-pads each
    response to a uniform length in [lo, hi]; ``prompt_pad_range=(lo, hi)``
    left-pads each prompt (same padding for all rows of a prompt).  Pad tokens
    get ``pad_id``.  ``shuffle`` scatters the rows with a seeded permutation."""
    rng = np.random.default_rng(seed)
    B = G * n
    L = P + R
    prompts = rng.integers(0, vocab, size=(G, P), dtype=np.int64)
    # distinct prompts (a repeat draw is astronomically unlikely, but cheap to rule out)
    for g in range(1, G):
        while any(np.array_equal(prompts[g], prompts[h]) for h in range(g)):
            prompts[g] = rng.integers(0, vocab, size=P, dtype=np.int64)
    responses = rng.integers(0, vocab, size=(B, R), dtype=np.int64)
    ids = np.empty((B, L), dtype=np.int64)
    mask = np.ones((B, L), dtype=np.uint8)
    prompt_pad = np.zeros(G, dtype=np.int64)
    if prompt_pad_range is not None:
        prompt_pad = rng.integers(prompt_pad_range[0], prompt_pad_range[1] + 1, size=G)
    for g in range(G):
        for j in range(n):
            b = g * n + j
            ids[b, :P] = prompts[g]
            ids[b, P:] = responses[b]
            if prompt_pad[g]:
                ids[b, :prompt_pad[g]] = pad_id
                mask[b, :prompt_pad[g]] = 0
    if resp_len_range is not None:
        lens = rng.integers(resp_len_range[0], resp_len_range[1] + 1, size=B)
        for b in range(B):
            ids[b, P + lens[b]:] = pad_id
            mask[b, P + lens[b]:] = 0
    if shuffle:
        perm = rng.permutation(B)
        ids = ids[perm]
        mask = mask[perm]
    has_mask = prompt_pad_range is not None or resp_len_range is not None
    pos = np.tile(np.arange(L, dtype=np.int64), (B, 1))
    if has_mask:
        pos = np.maximum(np.cumsum(mask, axis=1, dtype=np.int64) - 1, 0)
    return ids, (mask if has_mask else None), pos


def make_workload_batch(wl: Workload, index: int, shuffle=True):
    """The batch of a named workload, seeded with ``SEED_BASE + index``."""
    return make_batch(wl.G, wl.n, wl.P, wl.R, wl.vocab, SEED_BASE + index,
                      shuffle=shuffle, resp_len_range=wl.resp_len_range)


def make_qkv(T, Hq, Hkv, D, seed, with_grad=True):
    """Q, K, V (and dO) ~ N(0, 1) drawn directly in the packed layout
    ``[T, H, D]`` as float32 arrays; callers round to bf16 where needed."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, Hq, D), dtype=np.float32)
    k = rng.standard_normal((T, Hkv, D), dtype=np.float32)
    v = rng.standard_normal((T, Hkv, D), dtype=np.float32)
    do = rng.standard_normal((T, Hq, D), dtype=np.float32) if with_grad else None
    return q, k, v, do


def make_rows(B, L, W, seed):
    """A ``[B, L, W]`` float32 row tensor ~ N(0, 1) (hidden states)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, L, W), dtype=np.float32)


def bf16_round(x):
    """Round float32 to the nearest bfloat16 (ties to even), kept as float32."""
    a = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((a >> 16) & 1) + np.uint32(0x7FFF)
    out = ((a + r) & np.uint32(0xFFFF0000)).view(np.float32)
    return out.reshape(np.shape(x))
