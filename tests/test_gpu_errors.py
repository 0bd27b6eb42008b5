"""Bad data found on the GPU is reported through the workspace's error word, without a
fault: out-of-range block ids and context lengths. (No kernel waits on another, so no
case can hang.)"""
import numpy as np
import pytest
import torch

import decode_attention_paged_gqa_gb300 as da
from decode_attention_paged_gqa_gb300 import workloads as wl
from paged_cases import assert_close, make_case, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from decode_attention_paged_gqa_gb300 import build

    build.build()


def case():
    spec = wl.WorkloadSpec("err", 3, 8, 2, 128, "bf16", 600, 1800, seed=13)
    return make_case(spec)


def test_bad_block_id_sets_error_bit_and_other_sequences_stay_correct():
    c = case()
    good = run_oracle(c)
    c["bt"] = c["bt"].copy()
    c["bt"][1, 3] = c["num_blocks"] + 5  # sequence 1 points outside the pool
    p = None
    from paged_cases import params_for, to_device

    p = params_for(c)
    dev = to_device(c)
    ws = torch.empty(da.decode_attn_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    da.attach_workspace(p, ws)
    da.decode_attn_workspace_init(p)
    out = torch.empty((3, 8, 128), device="cuda")
    da.decode_attn_paged(dev["q"], dev["k"], dev["v"], None, None, None, None, dev["bt"], dev["lens"], out, p)
    err = da.decode_attn_get_device_error(p)
    assert err & da.DA_DEVERR_BLOCK_ID
    assert da.decode_attn_get_device_error(p) == 0  # read clears
    o = out.cpu().numpy()
    assert_close(o[[0, 2]], good[[0, 2]], "untouched sequences")


def test_bad_context_length_sets_error_bit():
    c = case()
    c["lens"] = c["lens"].copy()
    c["lens"][2] = 10 ** 6
    out = run_gpu(c, check_device_error=False)
    assert np.all(np.isfinite(out[:2]))
    from paged_cases import params_for

    c2 = case()
    c2["lens"] = c2["lens"].copy()
    c2["lens"][0] = -3
    p = params_for(c2)
    ws = torch.empty(da.decode_attn_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    da.attach_workspace(p, ws)
    da.decode_attn_workspace_init(p)
    from paged_cases import to_device

    dev = to_device(c2)
    out = torch.empty((3, 8, 128), device="cuda")
    da.decode_attn_paged(dev["q"], dev["k"], dev["v"], None, None, None, None, dev["bt"], dev["lens"], out, p)
    assert da.decode_attn_get_device_error(p) & da.DA_DEVERR_CONTEXT_LEN
    assert np.all(out[0].cpu().numpy() == 0)  # clamped to an empty sequence


def test_library_still_usable_after_bad_input():
    c = case()
    assert_close(run_gpu(c), run_oracle(c), "after errors")
