"""Pins for the oracle's mixed cache formats (attention.rs README, KV Cache Formats table):
"Turbo8" = FP8 E4M3 keys + 4-bit codebook values, "Turbo3" = 3-bit codebook keys + 4-bit
codebook values. The 3-bit codes are checked against an independent numpy bit packer and
attention against the rotated-basis route computed with library routines (the 8-level
codebook is pinned with the 16-level one in test_oracle_encoders.py)."""
import math

import numpy as np
import scipy.linalg
import torch

from test_oracle_attention import bf16_bits, bits_to_f64, paged, sdpa_ref

def pack_bits(codes, bits):
    """Independent packer: codes [..., D] -> bytes, code d at stream bits [bits*d, bits*d+bits)."""
    codes = np.asarray(codes, dtype=np.uint8)
    D = codes.shape[-1]
    stream = ((codes[..., :, None] >> np.arange(bits)) & 1).reshape(codes.shape[:-1] + (D * bits,))
    return np.packbits(stream.reshape(codes.shape[:-1] + (D * bits // 8, 8)), axis=-1, bitorder="little")[..., 0]


def test_three_bit_stream_layout(oracle):
    rng = np.random.default_rng(4)
    cb8 = oracle.lloyd_max(8, 1 / math.sqrt(128))[1]
    codes = rng.integers(0, 8, size=(5, 128))
    packed = pack_bits(codes, 3)
    assert packed.shape == (5, 48)
    scales = rng.random(5).astype(np.float32) + 0.5
    got = oracle.cb_dequant_rotated(3, packed, scales, cb8)
    assert np.array_equal(got, scales[:, None].astype(np.float64) * cb8.astype(np.float64)[codes])
    # the 4-bit layout is the same stream with b = 4 (low nibble first)
    cb16 = oracle.lloyd_max(16, 1 / math.sqrt(128))[1]
    codes4 = rng.integers(0, 16, size=(3, 128))
    got4 = oracle.cb_dequant_rotated(4, pack_bits(codes4, 4), scales[:3], cb16)
    assert np.array_equal(got4, scales[:3, None].astype(np.float64) * cb16.astype(np.float64)[codes4])


def test_three_bit_encoder_is_nearest_level(oracle):
    D = 128
    rng = np.random.default_rng(8)
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    cb8 = oracle.lloyd_max(8, 1 / math.sqrt(D))[1]
    x = rng.standard_normal((400, D)).astype(np.float32)
    packed, scale = oracle.cb_encode(3, x, sign, cb8)
    H = scipy.linalg.hadamard(D).astype(np.float64)
    u = (x.astype(np.float64) * sign) @ H.T / math.sqrt(D) / scale[:, None].astype(np.float64)
    ref_codes = np.abs(u[..., None] - cb8.astype(np.float64)).argmin(-1)
    assert np.array_equal(packed, pack_bits(ref_codes, 3))
    # round trip: 8-level distortion (0.03454 per unit-variance coordinate) times D sigma^2 = 1
    xh = oracle.cb_dequant(3, packed, scale, cb8, sign)
    rel = ((xh - x) ** 2).sum(1) / (x.astype(np.float64) ** 2).sum(1)
    assert 0.031 < rel.mean() < 0.038


def _mixed_case(oracle, fmt, seed):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D, lens = 2, 8, 2, 128, [90, 37]
    cb16 = oracle.lloyd_max(16, 1 / math.sqrt(D))[1]
    cb8 = oracle.lloyd_max(8, 1 / math.sqrt(D))[1]
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    xk = rng.standard_normal((B, Hkv, 90, D)).astype(np.float32)
    xv = rng.standard_normal((B, Hkv, 90, D)).astype(np.float32)
    q = bf16_bits(rng.standard_normal((B, Hq, D)))
    pv, sv = oracle.cb_encode(4, xv, sign, cb16)
    if fmt == "fp8k_cb4v":
        kcodes, ks = oracle.fp8_quantize(xk)
        kc, bt, _, _ = paged(kcodes, lens, 16, np.random.default_rng(1), 0)
        K_dense = torch.from_numpy(kcodes).view(torch.float8_e4m3fn).to(torch.float64) * float(ks)
        kscales = ks
        codebook = cb16
        K_rot = None
    else:
        pk, sk = oracle.cb_encode(3, xk, sign, cb8)
        kc, bt, _, _ = paged(pk, lens, 16, np.random.default_rng(1), 0)
        kscales = paged(sk[..., None], lens, 16, np.random.default_rng(1), 0)[0][..., 0]
        codebook = np.concatenate([cb8, cb16])
        K_rot = oracle.cb_dequant_rotated(3, pk, sk, cb8)
        K_dense = None
    vc, _, _, _ = paged(pv, lens, 16, np.random.default_rng(1), 0)
    vscales = paged(sv[..., None], lens, 16, np.random.default_rng(1), 0)[0][..., 0]
    out = oracle.decode_attention(q, kc, vc, bt, np.array(lens, np.int32), kv_format=fmt, num_kv_heads=Hkv,
                                  softmax_scale=1 / math.sqrt(D), k_scales=kscales, v_scales=vscales,
                                  codebook=codebook, sign_pattern=sign)
    H = scipy.linalg.hadamard(D).astype(np.float64)
    V_rot = oracle.cb_dequant_rotated(4, pv, sv, cb16)
    q64 = bits_to_f64(q).numpy()
    rot = lambda a: (a * sign) @ H.T / math.sqrt(D)        # noqa: E731  r = H diag(s) a / sqrt(D)
    unrot = lambda a: sign * (a @ H.T) / math.sqrt(D)      # noqa: E731  a = diag(s) H r / sqrt(D)
    if fmt == "fp8k_cb4v":
        # keys in the original basis, values rotated: attend with the original K, un-rotate the output
        o_rot = sdpa_ref(torch.from_numpy(q64), K_dense, torch.from_numpy(V_rot), lens, 1 / math.sqrt(D))
    else:
        o_rot = sdpa_ref(torch.from_numpy(rot(q64)), torch.from_numpy(K_rot), torch.from_numpy(V_rot), lens,
                         1 / math.sqrt(D))
    return out, unrot(o_rot)


def test_fp8_keys_codebook_values_matches_route(oracle):
    out, ref = _mixed_case(oracle, "fp8k_cb4v", 3)
    assert np.abs(out - ref).max() < 1e-12


def test_three_bit_keys_codebook_values_matches_route(oracle):
    out, ref = _mixed_case(oracle, "cb3k_cb4v", 5)
    assert np.abs(out - ref).max() < 1e-12
