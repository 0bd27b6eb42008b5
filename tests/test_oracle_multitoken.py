"""Pins for multi-token decode with a causal mask (attention.rs README, Features: causal
masking; speculative / multi-token-prediction decoding): T query tokens per sequence at
positions L-T .. L-1, token j attending positions <= L-T+j (and, with a window W, > L-T+j-W).
Checked against torch SDPA with an explicit boolean mask, against ordinary single-token
decode of each prefix, and for split-K invariance."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from test_oracle_attention import BF16_NAN, bf16_bits, bits_to_f64, paged


def multi_case(B, T, Hq, Hkv, D, lens, seed):
    rng = np.random.default_rng(seed)
    Lmax = max(lens)
    q = bf16_bits(rng.standard_normal((B, T, Hq, D)))
    Kd = bf16_bits(rng.standard_normal((B, Hkv, Lmax, D)))
    Vd = bf16_bits(rng.standard_normal((B, Hkv, Lmax, D)))
    kc, bt, _, _ = paged(Kd, lens, 16, np.random.default_rng(seed + 1), BF16_NAN)
    vc, _, _, _ = paged(Vd, lens, 16, np.random.default_rng(seed + 1), BF16_NAN)
    return dict(q=q, Kd=Kd, Vd=Vd, kc=kc, vc=vc, bt=bt, lens=np.array(lens, np.int32))


def run(oracle, c, Hkv, scale, **kw):
    return oracle.decode_attention(c["q"], c["kc"], c["vc"], c["bt"], c["lens"], kv_format="bf16",
                                   num_kv_heads=Hkv, softmax_scale=scale, **kw)


@pytest.mark.parametrize("T,window", [(2, 0), (4, 0), (3, 20), (8, 5)])
def test_multitoken_matches_sdpa_with_mask(oracle, T, window):
    B, Hq, Hkv, D, lens = 2, 8, 2, 64, [50, 9]
    c = multi_case(B, T, Hq, Hkv, D, lens, seed=T + window)
    ours = run(oracle, c, Hkv, 0.125, window=window)
    assert ours.shape == (B, T, Hq, D)
    q, K, V = bits_to_f64(c["q"]), bits_to_f64(c["Kd"]), bits_to_f64(c["Vd"])
    for b, L in enumerate(lens):
        pos = torch.arange(L - T, L)[:, None]
        t = torch.arange(L)[None, :]
        mask = t <= pos
        if window:
            mask &= t > pos - window
        ref = F.scaled_dot_product_attention(q[b].transpose(0, 1)[None], K[b][None, :, :L], V[b][None, :, :L],
                                             attn_mask=mask[None, None], scale=0.125, enable_gqa=True)
        assert np.abs(ours[b] - ref[0].transpose(0, 1).numpy()).max() < 1e-13


@pytest.mark.parametrize("window", [0, 300])
def test_each_query_token_equals_prefix_decode(oracle, window):
    B, T, Hq, Hkv, D, lens = 2, 4, 8, 2, 64, [1100, 600]
    c = multi_case(B, T, Hq, Hkv, D, lens, seed=5)
    multi = run(oracle, c, Hkv, 0.1, window=window, partition_size=512, split_threshold=1024)
    for jq in range(T):
        single = dict(c, q=c["q"][:, jq], lens=c["lens"] - (T - 1 - jq))
        ref = run(oracle, single, Hkv, 0.1, window=window)
        assert np.abs(multi[:, jq] - ref).max() < 1e-13


@pytest.mark.parametrize("psize", [1, 16, 100])
def test_multitoken_split_equals_unsplit(oracle, psize):
    c = multi_case(2, 4, 8, 2, 64, [700, 130], seed=psize)
    a = run(oracle, c, 2, 0.125, partition_size=0)
    b = run(oracle, c, 2, 0.125, partition_size=psize, split_threshold=1)
    assert np.abs(a - b).max() < 1e-12


def test_query_tokens_before_the_start_are_empty(oracle):
    c = multi_case(1, 4, 4, 1, 64, [2], seed=3)  # positions -2, -1, 0, 1
    out = run(oracle, c, 1, 0.125)
    assert np.all(out[0, :2] == 0)
    V = bits_to_f64(c["Vd"]).numpy()
    assert np.array_equal(out[0, 2], np.repeat(V[0, :, 0], 4, axis=0))


def test_multitoken_partition_grid_covers_all_queries():
    import oracle

    for L, T, W in [(5000, 4, 0), (5000, 4, 4096), (1030, 8, 1024), (3, 8, 0)]:
        b = oracle.partition_bounds(L, W, 512, 1024, query_len=T)
        first = max(0, L - T + 1 - W) if W else 0
        assert b[0][0] == first and b[-1][1] == L
        n = L - first
        assert len(b) == (-(-n // 512) if n >= 1024 else 1)
