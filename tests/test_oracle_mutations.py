"""The oracle's pins must catch plausible mistakes. Each case plants one mistake in a copy
of oracle/oracle.c (on the CPU), builds it, runs the pin tests against that build, and
requires at least one pin to fail. The planted copies live in a temporary directory."""
import os

import pytest

import oracle
import test_oracle_attention as A
import test_oracle_encoders as E
import test_oracle_alibi as AL
import test_oracle_multitoken as M
import test_oracle_mixed_formats as X

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text that occurs exactly once in oracle.c, replacement)
MUTATIONS = [
    ("gqa mapping interleaved", "int h = g * G + hh;", "int h = hh * j->Hkv + g;"),
    ("softmax scale dropped", "s[t - s0] = j->scale * acc;", "s[t - s0] = acc;"),
    ("softcap without the cap", "s[t - s0] = j->softcap * tanh(s[t - s0] / j->softcap);",
     "s[t - s0] = tanh(s[t - s0]);"),
    ("window off by one", "int a = window > 0 ? pos + 1 - window : 0;", "int a = window > 0 ? pos - window : 0;"),
    ("causal limit off by one", "int a = or_window_start(pos, j->window), e = pos + 1;",
     "int a = or_window_start(pos, j->window), e = pos + 2 < L ? pos + 2 : L;"),
    ("page slot off by one", "row = ((int64_t)phys * j->Hkv + g) * bs + t % bs;",
     "row = ((int64_t)phys * j->Hkv + g) * bs + (t + 1) % bs;"),
    ("K and V swapped", "const uint8_t* base = (const uint8_t*)(which ? j->v_cache : j->k_cache);",
     "const uint8_t* base = (const uint8_t*)(which ? j->k_cache : j->v_cache);"),
    ("partition weights dropped from the sum", "Lsum += lp[i] * w;", "Lsum += lp[i];"),
    ("partition outputs not rescaled", "out[d] += o[(int64_t)i * D + d] * w;", "out[d] += o[(int64_t)i * D + d];"),
    ("partition boundary off by one",
     "ends[p] = start + (p + 1) * partition_size < L ? start + (p + 1) * partition_size : L;",
     "ends[p] = start + (p + 1) * partition_size - 1 < L ? start + (p + 1) * partition_size - 1 : L;"),
    ("e4m3 exponent bias", "v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 9);"),
    ("e4m3 rounding half up", "r = nearbyint(q);", "r = floor(q + 0.5);"),
    ("e4m3 subnormal step", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("fp8 scale not applied", "double s = (double)(which ? j->v_scales[0] : j->k_scales[0]);", "double s = 1.0;"),
    ("bit order within a byte reversed", "v |= ((vec[s >> 3] >> (s & 7)) & 1) << i;",
     "v |= ((vec[s >> 3] >> (7 - (s & 7))) & 1) << i;"),
    ("un-rotation without the signs", "x[i] = (double)sign[i] * acc * inv;", "x[i] = acc * inv;"),
    ("hadamard transposed sign", "? -1.0 : 1.0;", "? 1.0 : -1.0;"),
    ("codebook ties to the upper index", "    if (d < bd) {", "    if (d <= bd) {"),
    ("codebook coordinates not normalised", "double u = scale > 0.0f ? r[i] / (double)scale : 0.0;",
     "double u = r[i];"),
    ("lloyd-max threshold not the midpoint", "for (i = 1; i < L; ++i) t[i] = 0.5 * (c[i - 1] + c[i]);",
     "for (i = 1; i < L; ++i) t[i] = c[i];"),
    ("bf16 decoded from the wrong half", "uint32_t w = (uint32_t)bits << 16;", "uint32_t w = (uint32_t)bits << 15;"),
    ("alibi bias with the wrong sign", "s[t - s0] += (double)j->alibi[h] * (double)(t - pos);",
     "s[t - s0] += (double)j->alibi[h] * (double)(pos - t);"),
    ("alibi slope of the kv head", "s[t - s0] += (double)j->alibi[h] * (double)(t - pos);",
     "s[t - s0] += (double)j->alibi[g] * (double)(t - pos);"),
    ("fp8 scale for a different maximum", "j.scale = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "j.scale = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    ("3-bit-key format decodes values with the key levels",
     "((j->fmt == OR_FMT_CB3K_CB4V && which) ? 8 : 0)", "0"),
    ("norm of the neighbouring token", "float sc = (which ? j->v_scales : j->k_scales)[row];",
     "float sc = (which ? j->v_scales : j->k_scales)[row ^ 1];"),
    ("query tokens in reverse order", "int64_t qi = ((int64_t)b * T + jq) * j->Hq + h;",
     "int64_t qi = ((int64_t)b * T + (T - 1 - jq)) * j->Hq + h;"),
]

PINS = [
    (A.test_bf16_matches_torch_sdpa, dict(D=64, Hq=8, Hkv=2, lens=[1, 37, 100])),
    (A.test_bf16_matches_torch_sdpa, dict(D=128, Hq=32, Hkv=8, lens=[77])),
    (A.test_fp8_matches_torch_sdpa, {}),
    (A.test_cb4_original_basis_equals_rotated_basis_route, {}),
    (A.test_split_k_equals_unsplit, dict(psize=100)),
    (A.test_single_key_returns_value_exactly, {}),
    (A.test_window_attends_last_tokens, dict(window=100)),
    (A.test_softcap_two_keys_closed_form, {}),
    (A.test_softcap_window_d256_matches_torch, {}),
    (A.test_partition_bounds_follow_pages, None),
    (M.test_multitoken_matches_sdpa_with_mask, dict(T=4, window=0)),
    (M.test_multitoken_matches_sdpa_with_mask, dict(T=3, window=20)),
    (AL.test_alibi_matches_sdpa_with_bias, dict(T=3, window=0, softcap=0.0)),
    (X.test_fp8_keys_codebook_values_matches_route, {}),
    (X.test_three_bit_keys_codebook_values_matches_route, {}),
    (E.test_fp8_quantize_scale_and_error_bound, {}),
    (E.test_e4m3_decode_fixed_points, {}),
    (E.test_e4m3_decode_matches_torch, {}),
    (E.test_e4m3_encode_matches_torch_cast, {}),
    (E.test_hadamard_is_sylvester, dict(D=16)),
    (E.test_lloyd_max_fixed_point_conditions, {}),
    (E.test_codebook_nearest_and_ties, "cb"),
    (E.test_cb4_nibble_order, "cb"),
    (E.test_cb4_roundtrip_distortion, "cb"),
    (E.test_cb4_rotation_direction_and_sign, "cb"),
]


def run_pins():
    """Names of the pins that fail against the currently loaded oracle build."""
    import math

    failed = []
    cb = None
    for fn, kw in PINS:
        try:
            if kw is None:
                fn()
            elif kw == "cb":
                if cb is None:
                    cb = oracle.lloyd_max(16, 1.0 / math.sqrt(128.0))[1]
                fn(oracle, cb)
            else:
                fn(oracle, **kw)
        except Exception:  # an assertion or an oracle error both count as caught
            failed.append(fn.__name__)
    return failed


def test_pins_pass_on_the_real_oracle():
    assert run_pins() == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique: {old!r}"
    src = tmp_path / "oracle_mut.c"
    src.write_text(text.replace(old, new))
    lib = oracle.compile_source(str(src), str(tmp_path / "liboracle_mut.so"))
    with oracle.library_override(lib):
        failed = run_pins()
    assert failed, f"no pin caught the planted mistake: {name}"
