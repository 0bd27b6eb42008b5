"""Test helpers: build a paged decode case from the seeded generators, encode its cache
with the ORACLE's encoders (test infrastructure), run it through the C-ABI library on the
GPU, and run the same bytes through the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from decode_attention_paged_gqa_gb300 import workloads as wl

# tolerance on the fp32 output against the fp64 oracle: max abs and relative L2
MAX_ABS = 2e-3
REL_L2 = 1e-3


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def make_case(spec: wl.WorkloadSpec, layout: wl.PagedLayout | None = None, sources: dict | None = None) -> dict:
    """All inputs of one call, on the CPU, in the library's layouts. `sources` may replace the
    generated fp32 K or V source ({"k": [num_blocks, Hkv, 16, D] tensor}) before encoding."""
    lay = layout or wl.make_layout(spec)
    nb = lay.num_blocks
    c = dict(spec=spec, lens=lay.context_lens, bt=lay.block_tables, num_blocks=nb, q=wl.make_query(spec),
             k_scales=None, v_scales=None, codebook=None, sign=None)
    k_side, v_side = oracle.SIDES[spec.kv_format]
    if "cb3" in (k_side, v_side) or "cb4" in (k_side, v_side):
        D = spec.head_dim
        cb16 = oracle.lloyd_max(16, 1.0 / math.sqrt(D))[1]
        cb8 = oracle.lloyd_max(8, 1.0 / math.sqrt(D))[1]
        c["codebook"] = torch.from_numpy(np.concatenate([cb8, cb16]) if k_side == "cb3" else cb16)
        c["sign"] = wl.sign_pattern(spec)
    sources = sources or {}
    for w, side in (("k", k_side), ("v", v_side)):
        if side == "bf16":
            c[w] = sources[w].to(torch.bfloat16) if w in sources else wl.kv_bf16(spec, w, nb)
            continue
        src = sources[w].float().numpy() if w in sources else wl.kv_source(spec, w, nb).numpy()
        if side == "fp8":
            codes, s = oracle.fp8_quantize(src)
            c[w] = torch.from_numpy(codes)
            c[w + "_scales"] = torch.tensor([s], dtype=torch.float32)
        else:
            bits = 3 if side == "cb3" else 4
            packed, scales = oracle.cb_encode(bits, src, c["sign"].numpy(), cb8 if bits == 3 else cb16)
            c[w] = torch.from_numpy(packed)
            c[w + "_scales"] = torch.from_numpy(scales)
    return c


def params_for(c: dict, **override):
    import decode_attention_paged_gqa_gb300 as da

    s = c["spec"]
    kw = dict(batch=s.batch, num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads, head_dim=s.head_dim,
              num_blocks=c["num_blocks"], max_blocks_per_seq=c["bt"].shape[1], max_context_len=s.ctx_max,
              kv_format=s.kv_format, softmax_scale=s.scale, softcap=s.softcap, window=s.window,
              partition_size=s.partition_size, split_threshold=s.split_threshold, block_size=s.block_size,
              query_len=s.query_len)
    kw.update(override)
    return da.make_params(**kw)


def to_device(c: dict, device="cuda") -> dict:
    d = {}
    for k in ("q", "k", "v", "k_scales", "v_scales", "codebook", "sign"):
        d[k] = None if c[k] is None else c[k].to(device)
    d["bt"] = torch.from_numpy(c["bt"]).to(device)
    d["lens"] = torch.from_numpy(c["lens"]).to(device)
    return d


def run_gpu(c: dict, dev: dict | None = None, params=None, check_device_error=True, **override) -> np.ndarray:
    """One decode_attn_paged call through the C ABI; returns out [B, Hq, D] (fp32, host)."""
    import decode_attention_paged_gqa_gb300 as da

    dev = dev or to_device(c)
    p = params or params_for(c, **override)
    ws = torch.empty(max(256, da.decode_attn_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    da.attach_workspace(p, ws)
    da.decode_attn_workspace_init(p)
    s = c["spec"]
    out = torch.full(tuple(c["q"].shape), float("nan"), dtype=torch.float32, device="cuda")
    da.decode_attn_paged(dev["q"], dev["k"], dev["v"], dev["k_scales"], dev["v_scales"], dev["codebook"],
                         dev["sign"], dev["bt"], dev["lens"], out, p)
    err = da.decode_attn_get_device_error(p)
    if check_device_error:
        assert err == 0, f"device error bits {err:#x}"
    return out.cpu().numpy()


def run_oracle(c: dict, select=None, **override) -> np.ndarray:
    s = c["spec"]
    kw = dict(kv_format=s.kv_format, num_kv_heads=s.num_kv_heads, softmax_scale=s.scale, softcap=s.softcap,
              window=s.window, partition_size=s.partition_size, split_threshold=s.split_threshold)
    kw.update(override)
    k = u16(c["k"]) if c["k"].dtype == torch.bfloat16 else c["k"].numpy()
    v = u16(c["v"]) if c["v"].dtype == torch.bfloat16 else c["v"].numpy()

    def np_or_none(t):
        return None if t is None else t.numpy()

    return oracle.decode_attention(u16(c["q"]), k, v, c["bt"], c["lens"], k_scales=np_or_none(c["k_scales"]),
                                   v_scales=np_or_none(c["v_scales"]), codebook=np_or_none(c["codebook"]),
                                   sign_pattern=np_or_none(c["sign"]), select=select, **kw)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    diff = gpu - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff)) / nref if nref > 0 else float(np.linalg.norm(diff))
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel
