"""decode_attn_paged_static_workspace -- the entry point for callers that cannot allocate
device memory (plugins inside frameworks that own every allocation, real-time loops that
must not call the allocator, callers without a CUDA allocator) -- must give the same output
as decode_attn_paged with a caller-provided workspace, call after call.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test. It passes both on its own in a fresh process and after
the other tests (the library's array keeps the previous call's contents; the entry point
clears what must start at zero)."""
import numpy as np
import pytest
import torch

import decode_attention_paged_gqa_gb300 as da
from decode_attention_paged_gqa_gb300 import workloads as wl
from paged_cases import MAX_ABS, REL_L2, assert_close, make_case, params_for, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from decode_attention_paged_gqa_gb300 import build

    build.build()


def static_call(c, out=None, dev=None):
    s = c["spec"]
    dev = dev or to_device(c)
    p = params_for(c)  # no workspace attached: the entry point uses the library's own array
    if out is None:
        out = torch.full(tuple(c["q"].shape), float("nan"), dtype=torch.float32, device="cuda")
    da.decode_attn_paged_static_workspace(dev["q"], dev["k"], dev["v"], dev["k_scales"], dev["v_scales"],
                                          dev["codebook"], dev["sign"], dev["bt"], dev["lens"], out, p)
    torch.cuda.synchronize()
    return out.cpu().numpy()


CASES = {
    # split and unsplit sequences, so the partials in the array are written and read
    "bf16": [dict(batch=4, hq=32, hkv=8, lo=300, hi=3000, seed=21), dict(batch=3, hq=16, hkv=8, lo=1000, hi=5000,
                                                                         seed=22)],
    "cb4": [dict(batch=4, hq=32, hkv=8, lo=300, hi=3000, seed=21), dict(batch=3, hq=16, hkv=8, lo=1000, hi=5000,
                                                                        seed=22)],
    # FP8: the reduce applies the per-tensor value scale
    "fp8": [dict(batch=4, hq=32, hkv=8, lo=300, hi=3000, seed=23), dict(batch=2, hq=8, hkv=2, lo=1500, hi=4000,
                                                                        seed=24)],
    # a sliding window with softcap, and two query tokens per sequence (multi-token decode)
    "bf16_window_softcap": [dict(batch=3, hq=16, hkv=8, lo=2000, hi=6000, seed=25, window=1500, softcap=30.0),
                            dict(batch=2, hq=8, hkv=4, lo=700, hi=3000, seed=26, window=1000, softcap=50.0)],
    "cb4_two_tokens": [dict(batch=3, hq=8, hkv=4, lo=300, hi=3000, seed=27, query_len=2),
                       dict(batch=2, hq=8, hkv=4, lo=1000, hi=2500, seed=28, query_len=2)],
}


def spec_for(name, fmt, d):
    return wl.WorkloadSpec(name, d["batch"], d["hq"], d["hkv"], 128, fmt, d["lo"], d["hi"], seed=d["seed"],
                           window=d.get("window", 0), softcap=d.get("softcap", 0.0), query_len=d.get("query_len", 1))


@pytest.mark.parametrize("case", sorted(CASES))
def test_static_workspace_matches_caller_workspace_twice(case):
    fmt = case.split("_")[0]
    for i, d in enumerate(CASES[case]):
        c = make_case(spec_for(f"noalloc_{case}_{i}", fmt, d))
        ref = run_gpu(c)
        got = static_call(c)
        max_abs, rel = assert_close(got, ref, f"{case} call {i}: static vs caller workspace")
        assert max_abs <= MAX_ABS and rel <= REL_L2


def test_static_workspace_call_allocates_nothing():
    """After a first (warm) call, a call through the static workspace leaves both torch's
    allocator and the device's free memory unchanged."""
    c = make_case(spec_for("noalloc_mem", "cb4", CASES["cb4"][1]))
    dev = to_device(c)
    out = torch.empty(tuple(c["q"].shape), dtype=torch.float32, device="cuda")
    first = static_call(c, out=out, dev=dev)
    torch.cuda.synchronize()
    allocated, free = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    second = static_call(c, out=out, dev=dev)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == allocated
    assert torch.cuda.mem_get_info()[0] == free
    assert np.array_equal(first, second)


def test_too_large_a_call_is_rejected():
    p = da.make_params(batch=64, num_q_heads=64, num_kv_heads=8, head_dim=256, num_blocks=1000,
                       max_blocks_per_seq=8192, max_context_len=131072, kv_format="bf16", softmax_scale=0.06)
    assert da.decode_attn_workspace_bytes(p) > 64 << 20
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_paged_static_workspace(256, 256, 256, None, None, None, None, 256, 256, 256, p)
    assert e.value.status == da._binding.DA_ERR_STATIC_WORKSPACE
