"""The C-ABI library without a GPU: it loads, exports every entry point the header
declares, and its host-side checks reject bad arguments before anything is enqueued."""
import ctypes
import os
import re

import pytest

import decode_attention_paged_gqa_gb300 as da
from decode_attention_paged_gqa_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def header_functions():
    text = open(os.path.join(ROOT, "include", "decode_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(decode_attn_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(da.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def base(**kw):
    d = dict(batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128, num_blocks=100, max_blocks_per_seq=64,
             max_context_len=1024, kv_format="bf16", softmax_scale=0.088)
    d.update(kw)
    return da.make_params(**d)


def test_workspace_bytes_and_partitions():
    p = base()
    assert da.decode_attn_max_partitions(p) == 2
    # err word + partials [B][Hq][P][D] f32 + max + sum, 256-byte aligned pieces
    n = da.decode_attn_workspace_bytes(p)
    assert n >= 4 * 32 * 2 * 128 * 4 + 2 * 4 * 32 * 2 * 4
    assert da.decode_attn_max_partitions(base(max_context_len=1023)) == 1
    assert da.decode_attn_max_partitions(base(max_context_len=32768)) == 64
    assert da.decode_attn_max_partitions(base(max_context_len=16384, window=4096)) == 8
    assert da.decode_attn_max_partitions(base(max_context_len=32768, partition_size=0)) == 1
    at_limit = base(max_context_len=8192 * 16, max_blocks_per_seq=8192, partition_size=16, split_threshold=1)
    assert da.decode_attn_max_partitions(at_limit) == 8192 and da.decode_attn_workspace_bytes(at_limit) > 0
    cb4 = da.decode_attn_workspace_bytes(base(kv_format="cb4"))
    assert cb4 >= n + 4 * 32 * 128 * 4  # plus the rotated queries


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=30), da._binding.DA_ERR_INVALID_ARG),     # Hq % Hkv != 0
    (dict(num_q_heads=24, num_kv_heads=2), da._binding.DA_ERR_UNSUPPORTED),  # G = 12
    (dict(head_dim=96), da._binding.DA_ERR_UNSUPPORTED),
    (dict(block_size=32), da._binding.DA_ERR_UNSUPPORTED),
    (dict(kv_format=7), da._binding.DA_ERR_INVALID_ARG),
    (dict(batch=-1), da._binding.DA_ERR_INVALID_ARG),
    (dict(softcap=-1.0), da._binding.DA_ERR_INVALID_ARG),
    (dict(softmax_scale=float("nan")), da._binding.DA_ERR_INVALID_ARG),
    (dict(window=-5), da._binding.DA_ERR_INVALID_ARG),
    (dict(partition_schedule=3), da._binding.DA_ERR_INVALID_ARG),
    (dict(partition_schedule=-1), da._binding.DA_ERR_INVALID_ARG),
    (dict(partitions_per_cta=65), da._binding.DA_ERR_INVALID_ARG),
    (dict(partitions_per_cta=-2), da._binding.DA_ERR_INVALID_ARG),
    (dict(max_context_len=1 << 30), da._binding.DA_ERR_UNSUPPORTED),  # more partitions than built
    (dict(max_context_len=8192 * 16 + 1, max_blocks_per_seq=8193, partition_size=16, split_threshold=1),
     da._binding.DA_ERR_UNSUPPORTED),  # 8193 partitions: one past the limit
])
def test_bad_params_are_rejected(kw, status):
    p = base(**kw)
    assert da.decode_attn_workspace_bytes(p) == 0
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_paged(16, 16, 16, None, None, None, None, 16, 16, 16, p, stream=0)
    assert e.value.status == status


@pytest.mark.parametrize("kw", [dict(head_dim=96), dict(num_q_heads=24, num_kv_heads=2), dict(block_size=32),
                                dict(max_context_len=1 << 30), dict(num_q_heads=30), dict(kv_format=7),
                                dict(softcap=-1.0), dict(query_len=9)])
def test_static_workspace_entry_returns_the_same_status(kw):
    """decode_attn_paged_static_workspace runs decode_attn_paged's checks first, so a rejected
    configuration gets the same status code from both entry points (and neither enqueues
    anything, so no GPU is needed)."""
    p = base(**kw)
    args = (256, 256, 256, None, None, None, None, 256, 256, 256, p)
    statuses = []
    for fn in (da.decode_attn_paged, da.decode_attn_paged_static_workspace):
        with pytest.raises(da.DecodeAttnError) as e:
            fn(*args, stream=0)
        statuses.append(e.value.status)
    assert statuses[0] == statuses[1] != da._binding.DA_ERR_WORKSPACE


def test_static_workspace_entry_checks_tensors_first():
    p = base()
    with pytest.raises(da.DecodeAttnError) as e:  # a NULL query: rejected before the array is touched
        da.decode_attn_paged_static_workspace(None, 256, 256, None, None, None, None, 256, 256, 256, p, stream=0)
    assert e.value.status == da._binding.DA_ERR_INVALID_ARG
    p = base(batch=0)  # nothing to do: returns at once, no CUDA call made
    da.decode_attn_paged_static_workspace(256, 256, 256, None, None, None, None, 256, 256, 256, p, stream=0)


def test_workspace_checks():
    p = base()
    with pytest.raises(da.DecodeAttnError) as e:  # no workspace
        da.decode_attn_paged(256, 256, 256, None, None, None, None, 256, 256, 256, p, stream=0)
    assert e.value.status == da._binding.DA_ERR_WORKSPACE
    p.workspace, p.workspace_bytes = 4096 + 128, 1 << 30  # misaligned
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_paged(256, 256, 256, None, None, None, None, 256, 256, 256, p, stream=0)
    assert e.value.status == da._binding.DA_ERR_WORKSPACE
    p.workspace, p.workspace_bytes = 4096, da.decode_attn_workspace_bytes(p) - 1  # too small
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_paged(256, 256, 256, None, None, None, None, 256, 256, 256, p, stream=0)
    assert e.value.status == da._binding.DA_ERR_WORKSPACE


def test_null_and_misaligned_tensors_are_rejected():
    p = base()
    p.workspace, p.workspace_bytes = 4096, da.decode_attn_workspace_bytes(p)
    cases = [
        (None, 256, 256, None, None, None, None, 256, 256, 256),          # q
        (256, 256, 256, None, None, None, None, None, 256, 256),          # block tables
        (256, 256 + 8, 256, None, None, None, None, 256, 256, 256),       # cache not 16-byte aligned
    ]
    for args in cases:
        with pytest.raises(da.DecodeAttnError) as e:
            da.decode_attn_paged(*args, p, stream=0)
        assert e.value.status == da._binding.DA_ERR_INVALID_ARG
    fp8 = base(kv_format="fp8")
    fp8.workspace, fp8.workspace_bytes = 4096, da.decode_attn_workspace_bytes(fp8)
    with pytest.raises(da.DecodeAttnError) as e:  # fp8 needs its scales
        da.decode_attn_paged(256, 256, 256, None, None, None, None, 256, 256, 256, fp8, stream=0)
    assert e.value.status == da._binding.DA_ERR_INVALID_ARG
    cb4 = base(kv_format="cb4")
    cb4.workspace, cb4.workspace_bytes = 4096, da.decode_attn_workspace_bytes(cb4)
    with pytest.raises(da.DecodeAttnError) as e:  # cb4 needs codebook and signs
        da.decode_attn_paged(256, 256, 256, 256, 256, None, None, 256, 256, 256, cb4, stream=0)
    assert e.value.status == da._binding.DA_ERR_INVALID_ARG
    p.alibi_slopes = 258  # ALiBi slopes not 4-byte aligned
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_paged(256, 256, 256, None, None, None, None, 256, 256, 256, p, stream=0)
    assert e.value.status == da._binding.DA_ERR_INVALID_ARG


def test_empty_batch_enqueues_nothing():
    p = base(batch=0)
    p.workspace, p.workspace_bytes = 4096, da.decode_attn_workspace_bytes(p)
    da.decode_attn_paged(256, 256, 256, None, None, None, None, 256, 256, 256, p, stream=0)  # no CUDA call made


def test_strerror():
    for s in range(-6, 1):
        assert da.decode_attn_strerror(s) != "unknown status"
    assert da.decode_attn_strerror(-99) == "unknown status"


@pytest.mark.parametrize("D", [64, 128, 256])
def test_library_codebook_equals_oracle_codebook(D):
    import math

    import numpy as np

    import oracle

    ours = np.array(da.decode_attn_codebook_lloyd_max(16, 1.0 / math.sqrt(D)), np.float32)
    ref = oracle.lloyd_max(16, 1.0 / math.sqrt(D))[1]
    assert np.array_equal(ours, ref)
    with pytest.raises(da.DecodeAttnError):
        da.decode_attn_codebook_lloyd_max(1, 1.0)


def test_params_keep_their_tensors_alive():
    """The params hold references to the workspace and slope tensors whose addresses they
    carry, so dropping the caller's names does not free memory a later call would use."""
    import gc
    import weakref

    import torch

    ws, slopes = torch.empty(1024, dtype=torch.uint8), torch.zeros(32, dtype=torch.float32)
    refs = weakref.ref(ws), weakref.ref(slopes)
    p = base(alibi_slopes=slopes)
    da.attach_workspace(p, ws)
    addr = ws.data_ptr()
    del ws, slopes
    gc.collect()
    assert all(r() is not None for r in refs)
    assert p.workspace == addr and p.workspace_bytes == 1024
