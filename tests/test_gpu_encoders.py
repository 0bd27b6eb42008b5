"""The library's cache writers on the GPU against the oracle's encoders: FP8 scale and
codes, 4-bit codebook norms and packed indices, all bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import decode_attention_paged_gqa_gb300 as da
from decode_attention_paged_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from decode_attention_paged_gqa_gb300 import build

    build.build()


@pytest.mark.parametrize("n,scale", [(1, 1.0), (1000, 3.0), (1 << 20, 1.0), (3_000_001, 1e-3)])
def test_fp8_encoder_bit_exact(n, scale):
    g = torch.Generator().manual_seed(n)
    x = torch.randn(n, generator=g) * scale
    x[::97] *= 50.0
    if n > 10:
        x[3] = 0.0
        x[5] = -0.0
    codes_ref, s_ref = oracle.fp8_quantize(x.numpy())
    xd = x.cuda()
    codes = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    da.decode_attn_encode_fp8(xd, n, codes, s)
    assert s.item() == s_ref
    assert np.array_equal(codes.cpu().numpy(), codes_ref)


def test_fp8_encoder_zero_tensor_and_repeat():
    x = torch.zeros(4096, device="cuda")
    codes = torch.full((4096,), 7, dtype=torch.uint8, device="cuda")
    s = torch.full((1,), 5.0, device="cuda")
    da.decode_attn_encode_fp8(x, 4096, codes, s)
    assert s.item() == 1.0 and int(codes.max()) == 0
    y = torch.randn(4096, device="cuda")
    da.decode_attn_encode_fp8(y, 4096, codes, s)  # the scale slot is reset each call
    ref_codes, ref_s = oracle.fp8_quantize(y.cpu().numpy())
    assert s.item() == ref_s and np.array_equal(codes.cpu().numpy(), ref_codes)


@pytest.mark.parametrize("D", [128, 256])
def test_cb4_encoder_bit_exact(D):
    spec = wl.WorkloadSpec("enc", 2, 8, 4, D, "cb4", 100, 300, seed=D)
    lay = wl.make_layout(spec)
    x = wl.kv_source(spec, "k", lay.num_blocks)
    x[0, 0, 0] = 0.0  # a zero vector
    sg = wl.sign_pattern(spec)
    cb = oracle.lloyd_max(16, 1.0 / math.sqrt(D))[1]
    packed_ref, scales_ref = oracle.cb4_encode(x.numpy(), sg.numpy(), cb)
    nvec = x.numel() // D
    packed = torch.empty(x.shape[:-1] + (D // 2,), dtype=torch.uint8, device="cuda")
    scales = torch.empty(x.shape[:-1], dtype=torch.float32, device="cuda")
    da.decode_attn_encode_cb4(x.cuda(), nvec, D, sg.cuda(), torch.from_numpy(cb).cuda(), packed, scales)
    assert np.array_equal(scales.cpu().numpy(), scales_ref)
    assert np.array_equal(packed.cpu().numpy(), packed_ref)


def test_cb4_encoder_rejects_bad_head_dim():
    with pytest.raises(da.DecodeAttnError):
        da.decode_attn_encode_cb4(256, 1, 96, 256, 256, 256, 256)


@pytest.mark.parametrize("D", [128, 256])
def test_three_bit_encoder_bit_exact(D):
    spec = wl.WorkloadSpec("enc3", 2, 8, 4, D, "cb3k_cb4v", 100, 300, seed=D + 1)
    lay = wl.make_layout(spec)
    x = wl.kv_source(spec, "k", lay.num_blocks)
    sg = wl.sign_pattern(spec)
    cb8 = oracle.lloyd_max(8, 1.0 / math.sqrt(D))[1]
    packed_ref, scales_ref = oracle.cb_encode(3, x.numpy(), sg.numpy(), cb8)
    nvec = x.numel() // D
    packed = torch.empty(x.shape[:-1] + (3 * D // 8,), dtype=torch.uint8, device="cuda")
    scales = torch.empty(x.shape[:-1], dtype=torch.float32, device="cuda")
    da.decode_attn_encode_codebook(x.cuda(), nvec, D, 3, sg.cuda(), torch.from_numpy(cb8).cuda(), packed, scales)
    assert np.array_equal(scales.cpu().numpy(), scales_ref)
    assert np.array_equal(packed.cpu().numpy(), packed_ref)


@pytest.mark.parametrize("D,bits,nvec", [(128, 4, 200_000), (256, 4, 40_000), (128, 3, 100_000), (256, 3, 40_000)])
def test_codebook_encoder_many_vectors_bit_exact(D, bits, nvec):
    """Enough vectors that the writer's fast path meets its fallbacks many times over (rotated
    coordinates within 1e-6 of a decision boundary, norms near a binary32 rounding boundary):
    every code and norm still equals the plain sequential fp64 evaluation's."""
    g = torch.Generator().manual_seed(D * 7 + bits)
    x = torch.randn(nvec, D, generator=g)
    x[1] = 0.0                      # a zero vector
    x[2] = 0.0
    x[2, 5] = 3.0                   # a one-hot vector (every rotated coordinate the same size)
    x[3:100] *= 1e-20               # tiny and huge norms
    x[100:200] *= 1e20
    sg = (torch.randint(0, 2, (D,), generator=g) * 2 - 1).to(torch.float32)
    cb = oracle.lloyd_max(1 << bits, 1.0 / math.sqrt(D))[1]
    packed_ref, scales_ref = oracle.cb_encode(bits, x.numpy(), sg.numpy(), cb)
    packed = torch.empty((nvec, D * bits // 8), dtype=torch.uint8, device="cuda")
    scales = torch.empty(nvec, dtype=torch.float32, device="cuda")
    da.decode_attn_encode_codebook(x.cuda(), nvec, D, bits, sg.cuda(), torch.from_numpy(cb).cuda(), packed, scales)
    assert np.array_equal(scales.cpu().numpy(), scales_ref)
    got = packed.cpu().numpy()
    assert np.array_equal(got, packed_ref), f"{int((got != packed_ref).sum())} bytes differ"


def test_codebook_encoder_unsorted_codebook():
    """A codebook that is not strictly increasing takes the plain evaluation for every
    coordinate: still the oracle's nearest level with ties to the lower index."""
    D, nvec = 128, 3000
    g = torch.Generator().manual_seed(5)
    x = torch.randn(nvec, D, generator=g)
    sg = (torch.randint(0, 2, (D,), generator=g) * 2 - 1).to(torch.float32)
    cb = oracle.lloyd_max(16, 1.0 / math.sqrt(D))[1][::-1].copy()  # decreasing
    cb[3] = cb[4]                                                     # and a repeated level
    packed_ref, scales_ref = oracle.cb_encode(4, x.numpy(), sg.numpy(), cb)
    packed = torch.empty((nvec, D // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(nvec, dtype=torch.float32, device="cuda")
    da.decode_attn_encode_codebook(x.cuda(), nvec, D, 4, sg.cuda(), torch.from_numpy(cb).cuda(), packed, scales)
    assert np.array_equal(scales.cpu().numpy(), scales_ref)
    assert np.array_equal(packed.cpu().numpy(), packed_ref)
