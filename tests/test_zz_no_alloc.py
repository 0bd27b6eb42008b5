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


def static_call(c):
    s = c["spec"]
    dev = to_device(c)
    p = params_for(c)  # no workspace attached: the entry point uses the library's own array
    out = torch.full((s.batch, s.num_q_heads, s.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    da.decode_attn_paged_static_workspace(dev["q"], dev["k"], dev["v"], dev["k_scales"], dev["v_scales"],
                                          dev["codebook"], dev["sign"], dev["bt"], dev["lens"], out, p)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("fmt", ["bf16", "cb4"])
def test_static_workspace_matches_caller_workspace_twice(fmt):
    # split and unsplit sequences, so the partials in the array are written and read
    first = make_case(wl.WorkloadSpec("noalloc1", 4, 32, 8, 128, fmt, 300, 3000, seed=21))
    second = make_case(wl.WorkloadSpec("noalloc2", 3, 16, 8, 128, fmt, 1000, 5000, seed=22))
    for c in (first, second):
        ref = run_gpu(c)
        got = static_call(c)
        max_abs, rel = assert_close(got, ref, f"{fmt} static vs caller workspace")
        assert max_abs <= MAX_ABS and rel <= REL_L2


def test_too_large_a_call_is_rejected():
    p = da.make_params(batch=64, num_q_heads=64, num_kv_heads=8, head_dim=256, num_blocks=1000,
                       max_blocks_per_seq=8192, max_context_len=131072, kv_format="bf16", softmax_scale=0.06)
    assert da.decode_attn_workspace_bytes(p) > 64 << 20
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_paged_static_workspace(256, 256, 256, None, None, None, None, 256, 256, 256, p)
    assert e.value.status == da._binding.DA_ERR_STATIC_WORKSPACE
