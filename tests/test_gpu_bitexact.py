"""Bit-exact checks of the integer and indexing work on the GPU: partition bounds, the
block-table gather, 4-bit unpacking and the dequantised values, compared with the oracle
integer for integer and bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import decode_attention_paged_gqa_gb300 as da
from decode_attention_paged_gqa_gb300 import workloads as wl
from paged_cases import make_case, params_for, run_gpu, run_oracle, to_device, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from decode_attention_paged_gqa_gb300 import build

    build.build()


def _ws(p):
    ws = torch.zeros(max(256, da.decode_attn_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    da.attach_workspace(p, ws)
    return ws


@pytest.mark.parametrize("window,psize,thresh,T", [(0, 512, 1024, 1), (4096, 512, 1024, 1), (1000, 100, 1, 1),
                                                   (0, 0, 1024, 1), (333, 16, 17, 1), (4096, 512, 1024, 4),
                                                   (1000, 100, 1, 8), (0, 512, 1024, 2)])
def test_partition_bounds_match_oracle(window, psize, thresh, T):
    lens = np.array(sorted(set(list(range(0, 2100, 7)) + [4095, 4096, 4097, 8191, 8192, 9000, 16384, 32768])),
                    np.int32)
    B = len(lens)
    spec = wl.WorkloadSpec("bounds", B, 8, 8, 128, "bf16", 0, 32768, seed=1, window=window, partition_size=psize,
                           split_threshold=thresh)
    p = da.make_params(batch=B, num_q_heads=8, num_kv_heads=8, head_dim=128, num_blocks=1,
                       max_blocks_per_seq=spec.max_blocks_per_seq, max_context_len=32768, kv_format="bf16",
                       softmax_scale=0.1, window=window, partition_size=psize, split_threshold=thresh, query_len=T)
    ws = _ws(p)
    P = da.decode_attn_max_partitions(p)
    bounds = torch.full((B, P, 2), -7, dtype=torch.int32, device="cuda")
    da.decode_attn_debug_partition_bounds(torch.from_numpy(lens).cuda(), bounds, p)
    got = bounds.cpu().numpy()
    assert da.decode_attn_get_device_error(p) == 0
    for b, L in enumerate(lens):
        ref = oracle.partition_bounds(int(L), window, psize, thresh, query_len=T)
        assert len(ref) <= P
        for i in range(P):
            exp = ref[i] if i < len(ref) else (-1, -1)
            assert tuple(got[b, i]) == exp, (int(L), i)


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("D", [128, 256])
def test_dequant_blocks_bitwise(fmt, D):
    spec = wl.WorkloadSpec("deq", 3, 8, 4, D, fmt, 200, 300, seed=D)
    c = make_case(spec)
    dev = to_device(c)
    p = params_for(c)
    ws = _ws(p)
    ids = torch.tensor([0, 5, c["num_blocks"] - 1, 2], dtype=torch.int32, device="cuda")
    out = torch.empty((4, spec.num_kv_heads, 16, D), dtype=torch.float32, device="cuda")
    sides = oracle.SIDES[fmt]
    for which, w in enumerate(("k", "v")):
        da.decode_attn_debug_dequant_blocks(dev[w], dev[w + "_scales"], dev["codebook"], ids, 4, which, out, p)
        got = out.cpu().numpy()
        sel = ids.cpu().numpy()
        side = sides[which]
        if side == "bf16":
            ref = oracle.bf16_decode(u16(c[w])[sel])
        elif side == "fp8":
            ref = oracle.e4m3_decode(c[w].numpy()[sel]) * float(c[w + "_scales"][0])
        else:
            bits = 3 if side == "cb3" else 4
            cb = c["codebook"].numpy()
            cb = cb[8:] if (fmt == "cb3k_cb4v" and which == 1) else cb
            ref = oracle.cb_dequant_rotated(bits, c[w].numpy()[sel], c[w + "_scales"].numpy()[sel], cb)
        # one fp32 rounding of an exact product on both sides
        assert np.array_equal(got, ref.astype(np.float32)), w
    assert da.decode_attn_get_device_error(p) == 0


def _dominant_key_case(fmt, L, window, j_list):
    """A batch where sequence i's key at position j_list[i] dominates every other score by
    far more than the fp32 exponent range, so softmax puts weight exactly 1 on it and the
    output is that token's value, bit for bit."""
    B = len(j_list)
    D, Hkv, G = 128, 2, 4
    spec = wl.WorkloadSpec(f"dom_{fmt}", B, Hkv * G, Hkv, D, fmt, L, L, seed=77, window=window)
    c = make_case(spec)
    q = torch.zeros_like(c["q"])
    q[..., 0] = 64.0
    c["q"] = q
    bt = c["bt"]
    # every other key gets 0 in coordinate 0, so its score is exactly 0
    c["k"][..., 0] = 0
    if fmt == "fp8":
        c["k_scales"][0] = 1.0
    for b, j in enumerate(j_list):
        phys = int(bt[b, j // 16])
        if fmt == "bf16":
            c["k"][phys, :, j % 16, 0] = 64.0  # score 64 * 64 / sqrt(128) = 362
        elif fmt == "fp8":
            c["k"][phys, :, j % 16, 0] = 0x7E  # e4m3 448: score 64 * 448 / sqrt(128) = 2534
        else:
            raise ValueError(fmt)
    return c


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
@pytest.mark.parametrize("window", [0, 700])
def test_dominant_key_gather_is_exact(fmt, window):
    L = 2600
    lo = L - window if window else 0
    # page edges, partition edges (512 from the first attended token), window edges
    js = sorted({lo, lo + 1, lo + 15, lo + 16, lo + 511, lo + 512, lo + 513, L - 1, L - 16, L - 17,
                 (lo + 1023) if lo + 1023 < L else L - 2})
    c = _dominant_key_case(fmt, L, window, js)
    out = run_gpu(c)
    ref = run_oracle(c)
    assert np.array_equal(out, ref.astype(np.float32))
    # and that is the value row of the dominant token
    for b, j in enumerate(js):
        phys = int(c["bt"][b, j // 16])
        if fmt == "bf16":
            v = c["v"][phys, :, j % 16].float().numpy()
        else:
            v = (oracle.e4m3_decode(c["v"][phys, :, j % 16].numpy()) * float(c["v_scales"][0])).astype(np.float32)
        assert np.array_equal(out[b], np.repeat(v, 4, axis=0))


def test_token_outside_window_is_not_read():
    # the token just before the window carries a huge key: it must have no effect
    L, W = 2600, 700
    c = make_case(wl.WorkloadSpec("win", 1, 8, 2, 128, "bf16", L, L, seed=5, window=W))
    q = torch.zeros_like(c["q"])
    q[..., 0] = 64.0
    c["q"] = q
    j = L - W - 1
    phys = int(c["bt"][0, j // 16])
    c["k"][phys, :, j % 16, 0] = 64.0
    out = run_gpu(c)
    assert np.abs(out - run_oracle(c)).max() < 2e-3
    assert not np.allclose(out[0, 0], c["v"][phys, 0, j % 16].float().numpy())


def test_single_token_returns_value_exactly():
    spec = wl.WorkloadSpec("one", 4, 32, 8, 128, "bf16", 1, 1, seed=9)
    c = make_case(spec)
    out = run_gpu(c)
    for b in range(4):
        phys = int(c["bt"][b, 0])
        v = c["v"][phys, :, 0].float().numpy()
        assert np.array_equal(out[b], np.repeat(v, 4, axis=0))
