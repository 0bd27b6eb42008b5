"""Pins for the oracle's paged GQA decode attention. Each check compares the oracle with
something other than itself: torch's scaled_dot_product_attention on a densely laid out
copy of the same keys and values (a library routine), plain Python loops on tiny inputs,
closed forms (uniform keys, a single key, an infinite softcap, a two-key softcap), and the
invariants of the method (any partition size gives the same result; permuting physical
blocks changes nothing). The pages' constants come from tests/golden/pages_constants.json."""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BF16_NAN = 0x7FC0


def bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def paged(dense, lens, bs, rng, fill, extra=3):
    """Lay dense per-sequence rows [B, Hkv, Lmax, *tail] into a shuffled page pool. Token
    slots past each length and unused blocks hold `fill` (NaN for bf16) so over-reads show."""
    B, Hkv, Lmax = dense.shape[:3]
    tail = dense.shape[3:]
    pages = [-(-int(L) // bs) for L in lens]
    nb = sum(pages) + extra
    perm = rng.permutation(nb)
    cache = np.full((nb, Hkv, bs) + tail, fill, dtype=dense.dtype)
    bt = np.full((B, max(1, max(pages))), -1, np.int32)
    off = 0
    for b in range(B):
        for p in range(pages[b]):
            phys = perm[off + p]
            bt[b, p] = phys
            lo, hi = p * bs, min(int(lens[b]), (p + 1) * bs)
            cache[phys, :, :hi - lo] = dense[b, :, lo:hi]
        off += pages[b]
    return cache, bt, perm, pages


def sdpa_ref(q64, K64, V64, lens, scale, window=0):
    """torch SDPA (fp64, CPU) per sequence over its attended rows; q [B,Hq,D], K/V [B,Hkv,Lmax,D]."""
    B, Hq, D = q64.shape
    out = torch.zeros((B, Hq, D), dtype=torch.float64)
    for b in range(B):
        L = int(lens[b])
        lo = max(0, L - window) if window else 0
        if L - lo <= 0:
            continue
        o = F.scaled_dot_product_attention(q64[b][None, :, None, :], K64[b][None, :, lo:L], V64[b][None, :, lo:L],
                                           scale=scale, enable_gqa=True)
        out[b] = o[0, :, 0, :]
    return out.numpy()


def rand_bf16_case(B, Hq, Hkv, D, lens, seed, bs=16):
    rng = np.random.default_rng(seed)
    Lmax = max(1, max(lens))
    q = bf16_bits(rng.standard_normal((B, Hq, D)))
    Kd = bf16_bits(rng.standard_normal((B, Hkv, Lmax, D)))
    Vd = bf16_bits(rng.standard_normal((B, Hkv, Lmax, D)))
    # the same permutation seed for K and V, so one block table serves both
    kc, bt, _, _ = paged(Kd, lens, bs, np.random.default_rng(seed + 1), BF16_NAN)
    vc, bt2, _, _ = paged(Vd, lens, bs, np.random.default_rng(seed + 1), BF16_NAN)
    assert np.array_equal(bt, bt2)
    return dict(q=q, Kd=Kd, Vd=Vd, kc=kc, vc=vc, bt=bt, lens=np.array(lens, np.int32))


def run(oracle, c, Hkv, scale, fmt="bf16", **kw):
    return oracle.decode_attention(c["q"], c["kc"], c["vc"], c["bt"], c["lens"], kv_format=fmt, num_kv_heads=Hkv,
                                   softmax_scale=scale, **kw)


# ------------------------------------------------------------------ library routine
@pytest.mark.parametrize("D,Hq,Hkv,lens", [(64, 8, 2, [1, 37, 100]), (128, 4, 4, [16, 15, 17]),
                                           (256, 16, 8, [300, 5]), (128, 32, 8, [77])])
def test_bf16_matches_torch_sdpa(oracle, D, Hq, Hkv, lens):
    c = rand_bf16_case(len(lens), Hq, Hkv, D, lens, seed=D + Hq)
    scale = 1 / math.sqrt(D)
    ours = run(oracle, c, Hkv, scale)
    ref = sdpa_ref(bits_to_f64(c["q"]), bits_to_f64(c["Kd"]), bits_to_f64(c["Vd"]), c["lens"], scale)
    assert np.abs(ours - ref).max() < 1e-13


def test_fp8_matches_torch_sdpa(oracle):
    rng = np.random.default_rng(21)
    B, Hq, Hkv, D, lens = 2, 8, 2, 128, [45, 130]
    q = bf16_bits(rng.standard_normal((B, Hq, D)))
    codes = rng.integers(0, 256, size=(2, B, Hkv, 130, D)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes in a cache
    kc, bt, _, _ = paged(codes[0], lens, 16, np.random.default_rng(5), 0)
    vc, _, _, _ = paged(codes[1], lens, 16, np.random.default_rng(5), 0)
    ks, vs = np.float32(0.0371), np.float32(0.00913)

    def dec(c):
        return torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64)

    ours = oracle.decode_attention(q, kc, vc, bt, np.array(lens, np.int32), kv_format="fp8", num_kv_heads=Hkv,
                                   softmax_scale=1 / math.sqrt(D), k_scales=ks, v_scales=vs)
    ref = sdpa_ref(bits_to_f64(q), dec(codes[0]) * float(ks), dec(codes[1]) * float(vs), lens, 1 / math.sqrt(D))
    assert np.abs(ours - ref).max() < 1e-13


def test_cb4_original_basis_equals_rotated_basis_route(oracle):
    """The oracle dequantises the codebook cache back to the original basis with a dense
    Hadamard matrix. The route the fast kernels take -- rotate q, attend in the rotated
    basis, un-rotate the output -- must give the same result (the rotation is orthogonal)."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, D, lens = 2, 8, 2, 128, [70, 33]
    _, cb, _ = oracle.lloyd_max(16, 1 / math.sqrt(D))
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    x = rng.standard_normal((2, B, Hkv, 70, D)).astype(np.float32)
    packed, scales = oracle.cb4_encode(x, sign, cb)
    kc, bt, _, _ = paged(packed[0], lens, 16, np.random.default_rng(6), 0)
    vc, _, _, _ = paged(packed[1], lens, 16, np.random.default_rng(6), 0)
    ksc, _, _, _ = paged(scales[0][..., None], lens, 16, np.random.default_rng(6), 0)
    vsc, _, _, _ = paged(scales[1][..., None], lens, 16, np.random.default_rng(6), 0)
    q = bf16_bits(rng.standard_normal((B, Hq, D)))
    scale = 1 / math.sqrt(D)
    ours = oracle.decode_attention(q, kc, vc, bt, np.array(lens, np.int32), kv_format="cb4", num_kv_heads=Hkv,
                                   softmax_scale=scale, k_scales=ksc[..., 0], v_scales=vsc[..., 0], codebook=cb,
                                   sign_pattern=sign)
    H = scipy.linalg.hadamard(D).astype(np.float64)
    q64 = bits_to_f64(q).numpy()
    q_rot = (q64 * sign) @ H.T / math.sqrt(D)
    K_rot = oracle.cb4_dequant_rotated(packed[0], scales[0], cb)
    V_rot = oracle.cb4_dequant_rotated(packed[1], scales[1], cb)
    o_rot = sdpa_ref(torch.from_numpy(q_rot), torch.from_numpy(K_rot), torch.from_numpy(V_rot), lens, scale)
    ref = sign * (o_rot @ H.T) / math.sqrt(D)
    assert np.abs(ours - ref).max() < 1e-12


# ------------------------------------------------------------------ plain loops
def test_matches_python_loops_tiny(oracle):
    rng = np.random.default_rng(2)
    B, Hq, Hkv, D, lens, bs = 2, 4, 2, 4, [5, 3], 2
    c = rand_bf16_case(B, Hq, Hkv, D, lens, seed=2, bs=bs)
    ours = oracle.decode_attention(c["q"], c["kc"], c["vc"], c["bt"], c["lens"], kv_format="bf16",
                                   num_kv_heads=Hkv, softmax_scale=0.7)
    q, K, V = bits_to_f64(c["q"]).tolist(), bits_to_f64(c["Kd"]).tolist(), bits_to_f64(c["Vd"]).tolist()
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            s = [0.7 * sum(q[b][h][d] * K[b][g][t][d] for d in range(D)) for t in range(lens[b])]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            for d in range(D):
                ref = sum(w[t] * V[b][g][t][d] for t in range(lens[b])) / sum(w)
                assert abs(ours[b, h, d] - ref) < 1e-14


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("psize", [1, 7, 16, 100, 512, 1000])
def test_split_k_equals_unsplit(oracle, psize):
    c = rand_bf16_case(3, 8, 2, 64, [1000, 513, 9], seed=41)
    full = run(oracle, c, 2, 0.125, partition_size=0)
    split = run(oracle, c, 2, 0.125, partition_size=psize, split_threshold=1)
    assert np.abs(split - full).max() < 1e-12


def test_block_permutation_invariance(oracle):
    c = rand_bf16_case(2, 8, 2, 128, [200, 61], seed=43)
    base = run(oracle, c, 2, 0.09)
    rng = np.random.default_rng(0)
    perm = rng.permutation(c["kc"].shape[0])  # new physical position of every block
    kc2 = np.empty_like(c["kc"])
    vc2 = np.empty_like(c["vc"])
    kc2[perm] = c["kc"]
    vc2[perm] = c["vc"]
    bt2 = np.where(c["bt"] >= 0, perm[np.maximum(c["bt"], 0)], -1).astype(np.int32)
    c2 = dict(c, kc=kc2, vc=vc2, bt=bt2)
    assert np.array_equal(run(oracle, c2, 2, 0.09), base)


def test_selected_rows_equal_full(oracle):
    c = rand_bf16_case(3, 8, 2, 64, [50, 1100, 7], seed=47)
    full = run(oracle, c, 2, 0.125, partition_size=512)
    sel = [(1, 7), (0, 0), (2, 3), (1, 2)]
    part = run(oracle, c, 2, 0.125, partition_size=512, select=sel)
    for i, (b, h) in enumerate(sel):
        assert np.array_equal(part[i], full[b, h])


# ------------------------------------------------------------------ closed forms
def test_uniform_keys_give_mean_of_values(oracle):
    c = rand_bf16_case(2, 8, 2, 64, [300, 41], seed=53)
    kc = c["kc"].copy()
    kc[...] = bf16_bits(np.full(64, 0.5))  # every key equal
    out = run(oracle, dict(c, kc=kc), 2, 0.125)
    V = bits_to_f64(c["Vd"]).numpy()
    for b, L in enumerate(c["lens"]):
        mean = V[b, :, :L].mean(axis=1)  # [Hkv, D]
        assert np.abs(out[b] - np.repeat(mean, 4, axis=0)).max() < 1e-13


def test_zero_query_gives_mean_of_values(oracle):
    c = rand_bf16_case(1, 4, 1, 64, [97], seed=59)
    q = np.zeros_like(c["q"])
    out = run(oracle, dict(c, q=q), 1, 0.125)
    V = bits_to_f64(c["Vd"]).numpy()
    assert np.abs(out[0] - V[0, :, :97].mean(axis=1)).max() < 1e-13


def test_single_key_returns_value_exactly(oracle):
    c = rand_bf16_case(2, 8, 2, 128, [1, 1], seed=61)
    out = run(oracle, c, 2, 0.0884)
    V = bits_to_f64(c["Vd"]).numpy()
    for b in range(2):
        assert np.array_equal(out[b], np.repeat(V[b, :, 0], 4, axis=0))


def test_empty_sequence_gives_zeros(oracle):
    g = json.load(open(os.path.join(GOLDEN, "pages_constants.json")))
    assert g["empty_context_output"]["value"] == "zeros"
    c = rand_bf16_case(3, 8, 2, 64, [0, 20, 0], seed=67)
    out = run(oracle, c, 2, 0.125)
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and np.all(np.isfinite(out[1])) and np.any(out[1] != 0)


def test_gqa_group_of_one_is_mha(oracle):
    c = rand_bf16_case(2, 4, 4, 64, [33, 90], seed=71)
    ours = run(oracle, c, 4, 0.125)
    ref = sdpa_ref(bits_to_f64(c["q"]), bits_to_f64(c["Kd"]), bits_to_f64(c["Vd"]), c["lens"], 0.125)
    assert np.abs(ours - ref).max() < 1e-13


# ------------------------------------------------------------------ window and softcap
@pytest.mark.parametrize("window", [1, 5, 16, 100, 333])
def test_window_attends_last_tokens(oracle, window):
    c = rand_bf16_case(3, 8, 2, 64, [400, 100, 3], seed=73)
    ours = run(oracle, c, 2, 0.125, window=window)
    ref = sdpa_ref(bits_to_f64(c["q"]), bits_to_f64(c["Kd"]), bits_to_f64(c["Vd"]), c["lens"], 0.125, window=window)
    assert np.abs(ours - ref).max() < 1e-13


def test_window_at_least_length_is_no_window(oracle):
    c = rand_bf16_case(2, 8, 2, 64, [400, 100], seed=79)
    assert np.array_equal(run(oracle, c, 2, 0.125, window=400), run(oracle, c, 2, 0.125))


def test_infinite_softcap_is_no_softcap(oracle):
    c = rand_bf16_case(2, 8, 2, 64, [100, 20], seed=83)
    a = run(oracle, c, 2, 0.125, softcap=1e30)
    b = run(oracle, c, 2, 0.125)
    assert np.abs(a - b).max() < 1e-14


def test_softcap_two_keys_closed_form(oracle):
    # two keys along q: raw scores s0, s1; with softcap c the weights are the logistic
    # function of c*tanh(s0/c) - c*tanh(s1/c)
    D, cap, scale = 64, 2.0, 0.5
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 2.0
    Kd = np.zeros((1, 1, 2, D)); Kd[0, 0, 0, 0] = 3.0; Kd[0, 0, 1, 0] = -1.0
    Vd = np.zeros((1, 1, 2, D)); Vd[0, 0, 0, 1] = 1.0; Vd[0, 0, 1, 2] = 1.0
    rng = np.random.default_rng(1)
    kc, bt, _, _ = paged(bf16_bits(Kd), [2], 16, rng, BF16_NAN)
    vc, _, _, _ = paged(bf16_bits(Vd), [2], 16, np.random.default_rng(1), BF16_NAN)
    out = oracle.decode_attention(bf16_bits(q), kc, vc, bt, np.array([2], np.int32), kv_format="bf16",
                                  num_kv_heads=1, softmax_scale=scale, softcap=cap)
    s0, s1 = cap * math.tanh(scale * 6.0 / cap), cap * math.tanh(scale * -2.0 / cap)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert abs(out[0, 0, 1] - w0) < 1e-15 and abs(out[0, 0, 2] - (1 - w0)) < 1e-15
    assert np.all(out[0, 0, 3:] == 0) and out[0, 0, 0] == 0


def test_softcap_window_d256_matches_torch(oracle):
    c = rand_bf16_case(2, 4, 2, 256, [700, 260], seed=89)
    ours = run(oracle, c, 2, 1 / 16, window=250, softcap=5.0, partition_size=64, split_threshold=128)
    q, K, V = bits_to_f64(c["q"]), bits_to_f64(c["Kd"]), bits_to_f64(c["Vd"])
    for b, L in enumerate(c["lens"]):
        lo = L - 250
        Kb = K[b].repeat_interleave(2, 0)[:, lo:L]  # [Hq, n, D]
        Vb = V[b].repeat_interleave(2, 0)[:, lo:L]
        s = torch.einsum("hd,hnd->hn", q[b], Kb) / 16
        s = 5.0 * torch.tanh(s / 5.0)
        ref = torch.einsum("hn,hnd->hd", torch.softmax(s, -1), Vb).numpy()
        assert np.abs(ours[b] - ref).max() < 1e-13


# ------------------------------------------------------------------ partition bounds
def test_partition_bounds_follow_pages():
    import oracle

    g = json.load(open(os.path.join(GOLDEN, "pages_constants.json")))
    P, T = g["partition_size"]["value"], g["split_threshold"]["value"]
    for window in (0, 4096, 1000):
        for L in list(range(0, 2100, 13)) + [4095, 4096, 4097, 8191, 8192, 16384, 32768]:
            b = oracle.partition_bounds(L, window, P, T)
            start = max(0, L - window) if window else 0
            n = L - start
            if n == 0:
                assert b == []
                continue
            expect = -(-n // P) if n >= T else 1
            assert len(b) == expect
            assert b[0][0] == start and b[-1][1] == L
            assert all(b[i][1] == b[i + 1][0] for i in range(len(b) - 1))
            assert all(0 < e - s <= (P if n >= T else n) for s, e in b)


def test_unsplit_when_partitioning_disabled():
    import oracle

    assert oracle.partition_bounds(32768, 0, 0, 1024) == [(0, 32768)]


def test_block_out_of_range_is_an_error(oracle):
    c = rand_bf16_case(1, 4, 1, 64, [40], seed=97)
    bt = c["bt"].copy()
    bt[0, 1] = c["kc"].shape[0]
    with pytest.raises(ValueError):
        run(oracle, dict(c, bt=bt), 1, 0.125)
