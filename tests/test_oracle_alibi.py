"""Pins for ALiBi slopes (attention.rs README, feature list: ALiBi slopes): the score of key
position t for a query at position pos gets slope_h * (t - pos) added after scaling (and
softcap), one slope per query head. Checked against torch SDPA given the same bias as an
explicit additive mask, with one and several query tokens, windows and a softcap; for
split-K invariance; and against the special cases a slope of 0 (no bias) and a single
attended key (the bias cannot matter)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from test_oracle_multitoken import multi_case, run
from test_oracle_attention import bits_to_f64


def geometric_slopes(Hq):
    # the usual ALiBi choice: 2^(-8 h / Hq) for h = 1 .. Hq
    return np.array([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], np.float32)


def sdpa_with_bias(c, lens, T, scale, slopes, window=0, softcap=0.0):
    q, K, V = bits_to_f64(c["q"]), bits_to_f64(c["Kd"]), bits_to_f64(c["Vd"])
    Hq, Hkv = q.shape[2], K.shape[1]
    out = []
    for b, L in enumerate(lens):
        pos = torch.arange(L - T, L, dtype=torch.float64)[:, None]
        t = torch.arange(L, dtype=torch.float64)[None, :]
        allowed = t <= pos
        if window:
            allowed &= t > pos - window
        Kb = K[b][:, :L].repeat_interleave(Hq // Hkv, dim=0)
        Vb = V[b][:, :L].repeat_interleave(Hq // Hkv, dim=0)
        qb = q[b].transpose(0, 1)  # [Hq, T, D]
        s = scale * qb @ Kb.transpose(1, 2)  # [Hq, T, L]
        if softcap:
            s = softcap * torch.tanh(s / softcap)
        bias = torch.from_numpy(slopes.astype(np.float64))[:, None, None] * (t - pos)[None]
        s = s + bias
        s = s.masked_fill(~allowed[None], float("-inf"))
        # the softmax of s through SDPA: unit scale, s as the additive mask, q . k = 0
        zq = torch.zeros_like(qb)
        o = F.scaled_dot_product_attention(zq[None], Kb[None], Vb[None], attn_mask=s[None], scale=1.0)
        out.append(o[0].transpose(0, 1).numpy())
    return np.stack(out)


@pytest.mark.parametrize("T,window,softcap", [(1, 0, 0.0), (1, 40, 0.0), (3, 0, 0.0), (2, 25, 30.0)])
def test_alibi_matches_sdpa_with_bias(oracle, T, window, softcap):
    B, Hq, Hkv, D, lens = 2, 8, 2, 64, [70, 33]
    c = multi_case(B, T, Hq, Hkv, D, lens, seed=40 + T + window)
    slopes = geometric_slopes(Hq)
    ours = run(oracle, c, Hkv, 0.125, window=window, softcap=softcap, alibi_slopes=slopes)
    ref = sdpa_with_bias(c, lens, T, 0.125, slopes, window=window, softcap=softcap)
    assert np.abs(ours - ref).max() < 1e-12


def test_alibi_sign_prefers_recent_keys(oracle):
    """With identical keys only the bias differs between positions: a positive slope puts the
    most weight on the query's own position, so the output moves toward the newest value."""
    B, T, Hq, Hkv, D, lens = 1, 1, 2, 1, 64, [200]
    c = multi_case(B, T, Hq, Hkv, D, lens, seed=3)
    c["kc"][:] = c["kc"][0:1, 0:1, 0:1, :]  # every key the same
    slopes = np.array([0.0, 1.0], np.float32)
    out = run(oracle, c, Hkv, 0.125, alibi_slopes=slopes)
    V = bits_to_f64(c["Vd"])[0, 0]
    # slope 0: the mean of the values; slope 1: weights e^(t - pos) -> mostly the last value
    assert np.abs(out[0, 0, 0] - V[:200].mean(0).numpy()).max() < 1e-12
    w = np.exp(np.arange(200) - 199.0)
    assert np.abs(out[0, 0, 1] - (w[:, None] * V[:200].numpy()).sum(0) / w.sum()).max() < 1e-12


def test_zero_slopes_are_no_alibi(oracle):
    c = multi_case(2, 2, 8, 2, 64, [90, 40], seed=8)
    base = run(oracle, c, 2, 0.1)
    assert np.array_equal(run(oracle, c, 2, 0.1, alibi_slopes=np.zeros(8, np.float32)), base)


@pytest.mark.parametrize("psize", [16, 512])
def test_alibi_split_equals_unsplit(oracle, psize):
    c = multi_case(2, 2, 8, 2, 64, [1500, 700], seed=12)
    slopes = geometric_slopes(8)
    whole = run(oracle, c, 2, 0.1, alibi_slopes=slopes, partition_size=0)
    split = run(oracle, c, 2, 0.1, alibi_slopes=slopes, partition_size=psize, split_threshold=1)
    assert np.abs(whole - split).max() < 1e-12


def test_single_key_ignores_alibi(oracle):
    c = multi_case(1, 1, 4, 1, 64, [1], seed=2)
    out = run(oracle, c, 1, 0.1, alibi_slopes=np.full(4, 5.0, np.float32))
    assert np.array_equal(out[0, 0], np.repeat(bits_to_f64(c["Vd"])[0, 0, 0][None].numpy(), 4, 0))  # [Hq, D]
