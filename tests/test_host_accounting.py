"""Host-side pieces the measurement rests on: the algorithmic byte count of a call (the
numerator of every GB/s figure) and the seeded paged layouts of the workloads."""
import numpy as np
import pytest

from decode_attention_paged_gqa_gb300 import metrics
from decode_attention_paged_gqa_gb300 import workloads as wl


@pytest.mark.parametrize("fmt,D,expect", [
    ("bf16", 128, 2 * 128 * 2), ("bf16", 256, 2 * 256 * 2), ("fp8", 128, 2 * 128),
    ("cb4", 128, 2 * (64 + 4)), ("fp8k_cb4v", 128, 128 + 64 + 4), ("cb3k_cb4v", 128, (48 + 4) + (64 + 4))])
def test_bytes_per_token_and_kv_head(fmt, D, expect):
    # K row + V row: element bytes x D, packed codes (D*bits/8 bytes) plus a 4-byte fp32 norm
    assert metrics.kv_bytes_per_token_head(fmt, D) == expect


def test_algorithmic_bytes_count_attended_tokens_one_by_one():
    lens = [0, 1, 15, 16, 17, 4095, 4096, 4097, 9000]
    for window in (0, 1, 16, 4096):
        tokens = 0
        for L in lens:
            start = max(0, L - window) if window else 0
            tokens += sum(1 for t in range(L) if t >= start)
        for fmt in metrics.FORMAT_BYTES:
            got = metrics.algorithmic_kv_bytes(lens, window, 8, fmt, 128)
            assert got == tokens * 8 * metrics.kv_bytes_per_token_head(fmt, 128)


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_layouts_are_valid_and_seeded(name):
    spec = wl.WORKLOADS[name]
    lay = wl.make_layout(spec)
    L, bt = lay.context_lens, lay.block_tables
    assert L.shape == (spec.batch,) and bt.shape == (spec.batch, spec.max_blocks_per_seq)
    assert L.min() >= spec.ctx_min and L.max() <= spec.ctx_max
    used = []
    for b in range(spec.batch):
        n = -(-int(L[b]) // spec.block_size)
        assert np.all(bt[b, :n] >= 0) and np.all(bt[b, :n] < lay.num_blocks) and np.all(bt[b, n:] == -1)
        used.extend(bt[b, :n].tolist())
    assert len(used) == len(set(used))  # no page is shared between sequences
    again = wl.make_layout(spec)
    assert np.array_equal(again.context_lens, L) and np.array_equal(again.block_tables, bt)


def test_described_batch_sizes():
    # the Llama-shaped batch's attended bytes, as its seeded lengths give them (a change of the
    # generator or of the accounting shows up here before it shows up in a GB/s figure)
    spec = wl.WORKLOADS["llama3_8b_bf16"]
    lay = wl.make_layout(spec)
    assert metrics.algorithmic_kv_bytes(lay.context_lens, 0, 8, "bf16", 128) == 1_075_286_016
    spec = wl.WORKLOADS["fp8_long_32k"]
    assert metrics.algorithmic_kv_bytes(wl.make_layout(spec).context_lens, 0, 8, "fp8", 128) == 16 * 32768 * 8 * 256
    spec = wl.WORKLOADS["gemma_window_softcap"]
    lay = wl.make_layout(spec)
    assert metrics.algorithmic_kv_bytes(lay.context_lens, 4096, 8, "bf16", 256) == 32 * 4096 * 8 * 1024
