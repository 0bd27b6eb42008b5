"""Pins for the oracle's cache encoders: E4M3, Sylvester Hadamard, Lloyd-Max codebook,
4-bit rotated-codebook quantise/pack. Each check uses something other than the oracle
itself: the format definition's fixed points, torch's float8 cast (run, not read), scipy's
Hadamard and numerical integration, the classical Gaussian Lloyd-Max table, closed forms."""
import json
import math
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.stats
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ E4M3
def test_e4m3_decode_fixed_points(oracle):
    # values fixed by the E4M3 definition (bias 7, 3 mantissa bits, subnormals, max 448)
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3F: 1.875,
             0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xB8: -1.0, 0xFE: -448.0}
    codes = np.array(list(table), dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    assert list(got) == [table[int(c)] for c in codes]
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    neg0 = oracle.e4m3_decode(np.array([0x80], np.uint8))[0]
    assert neg0 == 0.0 and math.copysign(1.0, neg0) < 0


def test_e4m3_decode_matches_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~finite)
    assert np.array_equal(ours[finite], ref[finite])
    # strictly increasing over the non-negative finite codes
    pos = ours[:0x7F]
    assert np.all(np.diff(pos) > 0)


def test_e4m3_roundtrip_all_finite_codes(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    assert np.array_equal(back, codes)  # +0 and -0 stay distinct


def _midpoints():
    pos = np.array([v for v in (np.arange(0x7F, dtype=np.uint8))], dtype=np.uint8)
    vals = torch.from_numpy(pos).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (vals[:-1] + vals[1:]) / 2  # exact in fp32: at most 5 significant bits
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(-np.inf))
    allv = np.concatenate([m32, up, dn])
    return np.concatenate([allv, -allv])


def test_e4m3_encode_matches_torch_cast(oracle):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, 2_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = np.concatenate([
        rng.standard_normal(5_000_000).astype(np.float32) * np.float32(60.0),
        rng.standard_normal(1_500_000).astype(np.float32) * np.float32(0.01),
        (rng.random(1_500_000).astype(np.float32) - np.float32(0.5)) * np.float32(900.0),
        bits[np.isfinite(bits)],  # every binary32 exponent, subnormals included
        _midpoints(),
        np.array([0.0, -0.0, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -11, 3 * 2.0 ** -10, 448.0, 463.99], np.float32),
    ]).astype(np.float32)
    x = x[np.abs(x) < 464.0]  # torch's cast turns |x| >= 464 into NaN; the oracle saturates there
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates(oracle):
    x = np.array([448.0, 449.0, 463.9, 464.0, 1000.0, 1e30, -500.0, np.inf, -np.inf], np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x7E] * 6 + [0xFE, 0x7E, 0xFE]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_fp8_quantize_scale_and_error_bound(oracle):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(200_000).astype(np.float32)
    codes, s = oracle.fp8_quantize(x)
    amax = np.float32(np.abs(x).max())
    assert s == np.float32(amax / np.float32(448.0))
    dec = oracle.e4m3_decode(codes)
    assert np.nanmax(np.abs(dec)) == 448.0
    # x / s (binary32) rounded once more to E4M3: half a grid step, relative 2^-4 above 2^-6,
    # absolute 2^-10 below it; the binary32 division adds at most one binary32 ulp
    y = (x / s).astype(np.float64)
    bound = np.where(np.abs(y) >= 2.0 ** -6, np.abs(y) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(dec - y) <= bound)
    assert np.array_equal(codes, oracle.e4m3_encode(x / s))


# ------------------------------------------------------------------ Hadamard
@pytest.mark.parametrize("D", [2, 16, 64, 128, 256])
def test_hadamard_is_sylvester(oracle, D):
    H = oracle.hadamard(D)
    assert np.array_equal(H, scipy.linalg.hadamard(D).astype(np.float64))
    assert np.array_equal(H @ H, D * np.eye(D))


# ------------------------------------------------------------------ Lloyd-Max codebook
def test_lloyd_max_fixed_point_conditions(oracle):
    sigma = 1.0 / math.sqrt(128.0)
    lv, cb, _ = oracle.lloyd_max(16, sigma)
    assert np.all(np.diff(lv) > 0)
    assert np.array_equal(lv, -lv[::-1])  # exactly symmetric
    assert np.array_equal(cb, lv.astype(np.float32))
    # centroid condition, checked by numerical integration (scipy quad), not the closed form
    t = np.concatenate([[-np.inf], (lv[:-1] + lv[1:]) / 2, [np.inf]])
    pdf = scipy.stats.norm(scale=sigma).pdf
    for i in range(16):
        mass = scipy.integrate.quad(pdf, t[i], t[i + 1], epsabs=1e-15, epsrel=1e-13)[0]
        mom = scipy.integrate.quad(lambda z: z * pdf(z), t[i], t[i + 1], epsabs=1e-15, epsrel=1e-13)[0]
        assert abs(mom / mass - lv[i]) < 1e-10 * sigma


def _gaussian_quantiser_distortion(pos):
    """Mean squared error of the symmetric quantiser of N(0, 1) with positive levels `pos`
    (sorted) and cell boundaries at the midpoints, in closed form, with its gradient. Over a
    cell [a, b] with level c: int (x - c)^2 phi = (1 + c^2)(Phi(b) - Phi(a)) - 2c(phi(a) - phi(b))
    + (a phi(a) - b phi(b)); d/dc = 2(c (Phi(b) - Phi(a)) - (phi(a) - phi(b))), the boundary
    terms cancelling at midpoints."""
    import scipy.stats

    c = np.concatenate([-pos[::-1], pos])
    t = np.concatenate([[-np.inf], (c[:-1] + c[1:]) / 2, [np.inf]])
    a, b = t[:-1], t[1:]
    Pa, Pb = scipy.stats.norm.cdf(a), scipy.stats.norm.cdf(b)
    fa, fb = scipy.stats.norm.pdf(a), scipy.stats.norm.pdf(b)
    afa = np.where(np.isfinite(a), a, 0.0) * fa  # x phi(x) -> 0 at +-inf
    bfb = np.where(np.isfinite(b), b, 0.0) * fb
    mse = np.sum((1 + c ** 2) * (Pb - Pa) - 2 * c * (fa - fb) + (afa - bfb))
    g = 2 * (c * (Pb - Pa) - (fa - fb))
    n = len(pos)
    return mse, g[n:] - g[:n][::-1]  # d/d pos_i: the level +pos_i and its mirror -pos_i


@pytest.mark.parametrize("levels", [8, 16])
def test_lloyd_max_is_the_distortion_minimum(oracle, levels):
    """The oracle's levels (a fixed-point iteration) against a different algorithm: direct
    minimisation of the closed-form distortion (scipy BFGS from evenly spaced levels)."""
    import scipy.optimize

    lv, _, _ = oracle.lloyd_max(levels, 1.0)
    x0 = np.linspace(0.2, 2.0, levels // 2)
    res = scipy.optimize.minimize(lambda p: _gaussian_quantiser_distortion(np.sort(p)), x0, jac=True,
                                  method="BFGS", options={"gtol": 1e-13, "maxiter": 10000})
    best = np.sort(res.x)
    assert np.abs(lv[levels // 2:] - best).max() < 1e-7
    assert abs(_gaussian_quantiser_distortion(lv[levels // 2:])[0] - res.fun) < 1e-13


# ------------------------------------------------------------------ 4-bit codebook encode
@pytest.fixture(scope="module")
def cb(oracle):
    return oracle.lloyd_max(16, 1.0 / math.sqrt(128.0))[1]


def test_codebook_nearest_and_ties(oracle, cb):
    for i in range(16):
        assert oracle.cb_nearest(float(cb[i]), cb) == i
    for i in range(15):
        mid = (float(cb[i]) + float(cb[i + 1])) / 2  # exact tie -> lower index
        assert oracle.cb_nearest(mid, cb) == i
        assert oracle.cb_nearest(mid + 1e-12, cb) == i + 1  # just past the tie
    assert oracle.cb_nearest(-10.0, cb) == 0 and oracle.cb_nearest(10.0, cb) == 15


def test_cb4_nibble_order(oracle, cb):
    # byte k holds coordinate 2k in the low nibble and 2k+1 in the high nibble
    packed = np.zeros((1, 64), np.uint8)
    packed[0, 0] = 0x21
    packed[0, 5] = 0xF0
    r = oracle.cb4_dequant_rotated(packed, np.array([2.0], np.float32), cb)[0]
    assert r[0] == 2.0 * float(cb[1]) and r[1] == 2.0 * float(cb[2])
    assert r[10] == 2.0 * float(cb[0]) and r[11] == 2.0 * float(cb[15])
    assert np.all(r[2:10] == 2.0 * float(cb[0]))


def test_cb4_rotation_direction_and_sign(oracle, cb):
    D = 128
    rng = np.random.default_rng(11)
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    H = scipy.linalg.hadamard(D).astype(np.float64)
    for k in (0, 5, 77, 127):
        x = np.zeros((1, D), np.float32)
        x[0, k] = 3.0
        packed, scale = oracle.cb4_encode(x, sign, cb)
        assert scale[0] == 3.0
        r = oracle.cb4_dequant_rotated(packed, scale, cb)[0] / 3.0
        # r = H diag(sign) x / (sqrt(D) ||x||) = sign_k H[:, k] / sqrt(D): every coordinate +-0.0884
        expect = sign[k] * H[:, k] / math.sqrt(D)
        assert np.all(np.sign(r) == np.sign(expect))
        assert np.all(np.abs(np.abs(r) - 1 / math.sqrt(D)) <= 0.02)


def test_cb4_roundtrip_distortion(oracle, cb):
    # x -> codes -> original basis: the relative squared error is the per-coordinate
    # Lloyd-Max distortion 0.009497 (unit-variance table value) times D * sigma^2 = 1
    D = 128
    rng = np.random.default_rng(5)
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    x = rng.standard_normal((4000, D)).astype(np.float32)
    packed, scale = oracle.cb4_encode(x, sign, cb)
    assert np.array_equal(scale, np.sqrt((x.astype(np.float64) ** 2).sum(1)).astype(np.float32))
    xh = oracle.cb4_dequant(packed, scale, cb, sign)
    rel = ((xh - x) ** 2).sum(1) / (x.astype(np.float64) ** 2).sum(1)
    assert 0.0085 < rel.mean() < 0.0105
    # the rotated-basis values are the same vector seen through an orthogonal map
    r = oracle.cb4_dequant_rotated(packed, scale, cb)
    H = scipy.linalg.hadamard(D).astype(np.float64)
    back = sign * (r @ H) / math.sqrt(D)
    assert np.allclose(back, xh, rtol=0, atol=1e-12)


def test_cb4_encode_is_nearest_level(oracle, cb):
    # every stored index is the nearest level to the fp64 rotated, normalised coordinate
    D = 128
    rng = np.random.default_rng(9)
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    x = rng.standard_normal((300, D)).astype(np.float32)
    packed, scale = oracle.cb4_encode(x, sign, cb)
    H = scipy.linalg.hadamard(D).astype(np.float64)
    u = (x.astype(np.float64) * sign) @ H.T / math.sqrt(D) / scale[:, None].astype(np.float64)
    idx = np.empty((300, D), np.int64)
    idx[:, 0::2] = packed & 15
    idx[:, 1::2] = packed >> 4
    dist = np.abs(u[..., None] - cb.astype(np.float64)[None, None, :])
    assert np.array_equal(idx, dist.argmin(-1))


def test_compression_ratios_match_pages():
    g = json.load(open(os.path.join(GOLDEN, "pages_constants.json")))["compression_vs_bf16"]
    D = 128
    bf16 = 2 * D
    fp8 = D
    cb4 = D // 2 + 4  # packed nibbles plus one fp32 norm per vector
    assert abs(bf16 / fp8 - g["values"]["fp8_e4m3"]) <= g["printed_precision"]
    assert abs(bf16 / cb4 - g["values"]["turbo4_4bitk_4bitv"]) <= g["printed_precision"] + 0.02
    # the mixed format (FP8 K, 4-bit V) of the same table
    assert abs(2 * bf16 / (fp8 + cb4) - g["values"]["turbo8_fp8k_4bitv"]) <= g["printed_precision"]
