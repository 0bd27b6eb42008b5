"""Byte accounting for the decode-attention roofline.

Algorithmic KV bytes of one call count exactly the attended tokens' K and V rows:
    sum_b min(L_b, window or L_b) * Hkv * (bytes of one K row + one V row)
with, per token and kv head, bf16: 2 * 2D bytes; FP8 E4M3: 2 * D; 4-bit codebook:
2 * (D / 2 + 4) (packed nibbles plus the fp32 norm); FP8 K + 4-bit V: D + D / 2 + 4;
3-bit K + 4-bit V: 3D / 8 + 4 + D / 2 + 4. Queries, outputs, partials, block
tables and per-tensor scales are not counted (they are < 1% of the traffic here).
"""
from __future__ import annotations

import numpy as np

FORMAT_BYTES = {
    "bf16": lambda D: 2 * 2 * D,
    "fp8": lambda D: 2 * D,
    "cb4": lambda D: 2 * (D // 2 + 4),
    "fp8k_cb4v": lambda D: D + (D // 2 + 4),
    "cb3k_cb4v": lambda D: (3 * D // 8 + 4) + (D // 2 + 4),
}


def kv_bytes_per_token_head(fmt: str, D: int) -> int:
    return FORMAT_BYTES[fmt](D)


def attended_tokens(context_lens, window: int = 0) -> int:
    L = np.asarray(context_lens, dtype=np.int64)
    if window > 0:
        L = np.minimum(L, window)
    return int(L.sum())


def algorithmic_kv_bytes(context_lens, window: int, num_kv_heads: int, fmt: str, D: int) -> int:
    return attended_tokens(context_lens, window) * num_kv_heads * kv_bytes_per_token_head(fmt, D)
