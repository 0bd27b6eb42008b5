"""Seeded synthetic inputs for single-token paged GQA decode attention.

This module only draws random numbers and lays them out as a paged KV cache: context
lengths, block tables, queries, per-block K/V source values and the random sign pattern
of the codebook format. It holds none of the attention arithmetic and none of the cache
encoders (FP8 and 4-bit codebook encoding happen in the consumers). Both the CUDA path
and the CPU oracle are fed from here; nothing else is shared between them.

Every tensor is drawn on the CPU with its own ``torch.Generator`` seed, so every consumer
sees identical bytes. K/V sources are drawn in chunks of ``CHUNK_BLOCKS`` physical blocks,
each chunk from its own seed, so any range of blocks can be regenerated on its own.

Workloads (named by what they are; shapes follow the decode batches described for this
attention: a Llama-3-8B-shaped BF16 batch, an FP8 long-context batch, a Gemma-style
sliding-window batch with softcap, and a 4-bit rotated-codebook batch):
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

CHUNK_BLOCKS = 256


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_format: str             # "bf16" | "fp8" | "cb4" | "fp8k_cb4v" | "cb3k_cb4v"
    ctx_min: int               # context lengths are uniform integers in [ctx_min, ctx_max]
    ctx_max: int
    seed: int
    block_size: int = 16
    window: int = 0            # 0: attend everything; else only the last `window` tokens
    softcap: float = 0.0       # 0: off; else scores become softcap * tanh(s / softcap)
    softmax_scale: Optional[float] = None  # default 1 / sqrt(head_dim)
    partition_size: int = 512
    split_threshold: int = 1024
    pool_blocks: Optional[int] = None      # fixed physical pool size (else the sum of pages needed)
    query_len: int = 1         # query tokens per sequence (the last ones of the context)

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.ctx_max // self.block_size)


WORKLOADS = {
    # batch 1, 8 query heads / 2 KV heads, D 128, 1024 tokens, 64 physical blocks
    "tiny_bf16": WorkloadSpec("tiny_bf16", 1, 8, 2, 128, "bf16", 1024, 1024, seed=1001, pool_blocks=64),
    # Llama-3-8B-shaped decode batch: 64 sequences, 32/8 heads, D 128, lengths U[512, 8192]
    "llama3_8b_bf16": WorkloadSpec("llama3_8b_bf16", 64, 32, 8, 128, "bf16", 512, 8192, seed=1002),
    # FP8 E4M3 cache, 16 sequences of 32768 tokens, 32/8 heads, D 128
    "fp8_long_32k": WorkloadSpec("fp8_long_32k", 16, 32, 8, 128, "fp8", 32768, 32768, seed=1003),
    # Gemma-style: 32 sequences, 16/8 heads, D 256, lengths U[4096, 16384], window 4096, softcap 50
    "gemma_window_softcap": WorkloadSpec("gemma_window_softcap", 32, 16, 8, 256, "bf16", 4096, 16384, seed=1004,
                                         window=4096, softcap=50.0, softmax_scale=1.0 / 16.0),
    # 4-bit rotated-codebook cache, 32 sequences of 32768 tokens, 32/8 heads, D 128
    "cb4_long_32k": WorkloadSpec("cb4_long_32k", 32, 32, 8, 128, "cb4", 32768, 32768, seed=1005),
    # the same batch with FP8 keys + 4-bit values, and with 3-bit keys + 4-bit values
    "fp8k_cb4v_long_32k": WorkloadSpec("fp8k_cb4v_long_32k", 32, 32, 8, 128, "fp8k_cb4v", 32768, 32768, seed=1006),
    "cb3k_cb4v_long_32k": WorkloadSpec("cb3k_cb4v_long_32k", 32, 32, 8, 128, "cb3k_cb4v", 32768, 32768, seed=1007),
    # smaller batches of spread lengths (how well the work is spread over the SMs): 16 Llama-shaped
    # BF16 sequences of U[512, 8192] tokens, and 32 4-bit sequences of U[1, 32768] tokens
    "llama3_8b_bf16_b16": WorkloadSpec("llama3_8b_bf16_b16", 16, 32, 8, 128, "bf16", 512, 8192, seed=1008),
    "cb4_spread_32k": WorkloadSpec("cb4_spread_32k", 32, 32, 8, 128, "cb4", 1, 32768, seed=1009),
    # multi-token decode (4 draft tokens per sequence) on the Llama-shaped batch: 16 (query
    # token, head) pairs per kv head, two column groups
    "llama3_8b_bf16_t4": WorkloadSpec("llama3_8b_bf16_t4", 64, 32, 8, 128, "bf16", 512, 8192, seed=1002,
                                      query_len=4),
}


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)


def _sub_seed(spec_seed: int, *parts: int) -> int:
    s = int(spec_seed)
    for p in parts:
        s = (s * 1_000_003 + int(p) + 7) % (1 << 61)
    return s


@dataclasses.dataclass
class PagedLayout:
    context_lens: np.ndarray   # int32 [B]
    block_tables: np.ndarray   # int32 [B, max_blocks_per_seq]; unused slots are -1
    num_blocks: int            # physical blocks in the pool


def make_layout(spec: WorkloadSpec, lens=None) -> PagedLayout:
    """Context lengths and block tables. Sequence b needs ceil(L_b / bs) pages; the pool
    holds at least the sum of those, and one seeded permutation of the pool is dealt out
    to the sequences in order. `lens` gives explicit context lengths instead of drawing them."""
    g = _gen(_sub_seed(spec.seed, 1))
    B, bs = spec.batch, spec.block_size
    if lens is not None:
        lens = torch.as_tensor(np.asarray(lens), dtype=torch.int64)
        assert lens.shape == (B,) and (B == 0 or int(lens.max()) <= spec.ctx_max)
    elif spec.ctx_min == spec.ctx_max:
        lens = torch.full((B,), spec.ctx_min, dtype=torch.int64)
    else:
        lens = torch.randint(spec.ctx_min, spec.ctx_max + 1, (B,), generator=g)
    pages = (lens + bs - 1) // bs
    need = int(pages.sum())
    pool = max(need, spec.pool_blocks or 0, 1)
    perm = torch.randperm(pool, generator=_gen(_sub_seed(spec.seed, 2))).to(torch.int32)
    tables = torch.full((B, spec.max_blocks_per_seq), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(pages[b])
        tables[b, :n] = perm[off:off + n]
        off += n
    return PagedLayout(lens.to(torch.int32).numpy(), tables.numpy(), pool)


def make_query(spec: WorkloadSpec) -> torch.Tensor:
    """q [B, Hq, D] (or [B, T, Hq, D] with T = query_len > 1), iid N(0, 1) rounded to bf16."""
    g = _gen(_sub_seed(spec.seed, 3))
    shape = (spec.batch,) + ((spec.query_len,) if spec.query_len > 1 else ()) + (spec.num_q_heads, spec.head_dim)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def kv_source(spec: WorkloadSpec, which: str, num_blocks: int, first: int = 0, count: Optional[int] = None):
    """fp32 K or V source values [count, Hkv, bs, D] of physical blocks [first, first+count),
    iid N(0, 1). Drawn chunk by chunk (CHUNK_BLOCKS blocks per seed)."""
    if count is None:
        count = num_blocks - first
    tag = {"k": 11, "v": 12}[which]
    shape_tail = (spec.num_kv_heads, spec.block_size, spec.head_dim)
    out = torch.empty((count,) + shape_tail, dtype=torch.float32)
    c0, c1 = first // CHUNK_BLOCKS, (first + count + CHUNK_BLOCKS - 1) // CHUNK_BLOCKS
    for c in range(c0, c1):
        lo, hi = c * CHUNK_BLOCKS, min((c + 1) * CHUNK_BLOCKS, num_blocks)
        chunk = torch.randn((hi - lo,) + shape_tail, generator=_gen(_sub_seed(spec.seed, tag, c)))
        a, b = max(lo, first), min(hi, first + count)
        out[a - first:b - first] = chunk[a - lo:b - lo]
    return out


def kv_bf16(spec: WorkloadSpec, which: str, num_blocks: int) -> torch.Tensor:
    """BF16 cache [num_blocks, Hkv, bs, D]: the N(0, 1) source rounded to bf16."""
    return kv_source(spec, which, num_blocks).to(torch.bfloat16)


def sign_pattern(spec: WorkloadSpec) -> torch.Tensor:
    """Fixed random +-1 vector of length D (fp32) for the codebook format's rotation."""
    g = _gen(_sub_seed(spec.seed, 4))
    return (torch.randint(0, 2, (spec.head_dim,), generator=g) * 2 - 1).to(torch.float32)


def scaled(spec: WorkloadSpec, **changes) -> WorkloadSpec:
    """A copy of a workload with some fields changed (smaller batch, other lengths, ...)."""
    return dataclasses.replace(spec, **changes)
