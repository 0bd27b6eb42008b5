"""ctypes binding of libdecode_attn (include/decode_attn.h), argument marshalling only.

Every entry point keeps the C name and argument order. Tensor arguments may be torch
tensors (their data_ptr() is passed), raw integer device addresses, or None for a NULL
pointer. ``stream`` may be None (torch's current stream), a torch.cuda.Stream, or a raw
cudaStream_t integer. A non-zero status raises DecodeAttnError. There is no fallback: if
the compiled library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdecode_attn.so")

DA_KV_BF16, DA_KV_FP8_E4M3, DA_KV_CB4, DA_KV_FP8K_CB4V, DA_KV_CB3K_CB4V = 0, 1, 2, 3, 4
KV_FORMATS = {"bf16": DA_KV_BF16, "fp8": DA_KV_FP8_E4M3, "cb4": DA_KV_CB4, "fp8k_cb4v": DA_KV_FP8K_CB4V,
              "cb3k_cb4v": DA_KV_CB3K_CB4V}
DA_OK, DA_ERR_INVALID_ARG, DA_ERR_UNSUPPORTED, DA_ERR_WORKSPACE, DA_ERR_LAUNCH, DA_ERR_CUDA = 0, -1, -2, -3, -4, -5
DA_ERR_STATIC_WORKSPACE = -6
DA_DEVERR_BLOCK_ID, DA_DEVERR_CONTEXT_LEN, DA_DEVERR_TIMEOUT, DA_DEVERR_SMEM_LAYOUT = 0x1, 0x2, 0x4, 0x8


class DecodeAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {decode_attn_strerror(status)} ({status})")
        self.status = status


class da_params(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("query_len", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("max_context_len", ctypes.c_int32),
        ("kv_format", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("window", ctypes.c_int32),
        ("partition_size", ctypes.c_int32),
        ("split_threshold", ctypes.c_int32),
        ("partition_schedule", ctypes.c_int32),
        ("partitions_per_cta", ctypes.c_int32),
        ("alibi_slopes", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


def make_params(*, batch, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq, max_context_len,
                kv_format, softmax_scale, softcap=0.0, window=0, partition_size=512, split_threshold=1024,
                block_size=16, query_len=1, partition_schedule=0, partitions_per_cta=0,
                alibi_slopes=None, workspace=None) -> da_params:
    p = da_params()
    p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim = batch, num_q_heads, num_kv_heads, head_dim
    p.query_len = int(query_len)
    p.block_size, p.num_blocks, p.max_blocks_per_seq, p.max_context_len = (block_size, num_blocks,
                                                                           max_blocks_per_seq, max_context_len)
    p.kv_format = KV_FORMATS[kv_format] if isinstance(kv_format, str) else int(kv_format)
    p.softmax_scale, p.softcap, p.window = float(softmax_scale), float(softcap), int(window)
    p.partition_size, p.split_threshold = int(partition_size), int(split_threshold)
    p.partition_schedule, p.partitions_per_cta = int(partition_schedule), int(partitions_per_cta)
    p.alibi_slopes = _ptr(alibi_slopes)  # a device tensor of Hq float32 slopes, or None
    p._alibi_ref = alibi_slopes  # the params hold the tensors they point at
    if workspace is not None:
        attach_workspace(p, workspace)
    return p


def attach_workspace(p: da_params, workspace) -> da_params:
    """Point the params at a device buffer (torch tensor) used as the call's workspace. The
    params keep a reference to the tensor, so it lives at least as long as they do."""
    p.workspace = workspace.data_ptr()
    p.workspace_bytes = workspace.numel() * workspace.element_size()
    p._workspace_ref = workspace
    return p


_lib = None
_lock = threading.Lock()


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libdecode_attn is not built ({LIB_PATH} missing); "
                                   "run decode_attention_paged_gqa_gb300.build.build()")
            lib = ctypes.CDLL(LIB_PATH)
            P, I, PP = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(da_params)
            call = [P, P, P, P, P, P, P, P, P, P, PP, P]
            sigs = {
                "decode_attn_workspace_bytes": (ctypes.c_size_t, [PP]),
                "decode_attn_workspace_init": (I, [PP, P]),
                "decode_attn_paged": (I, call),
                "decode_attn_paged_static_workspace": (I, call),
                "decode_attn_rotate_q": (I, call),
                "decode_attn_partition": (I, call),
                "decode_attn_reduce": (I, call),
                "decode_attn_get_device_error": (I, [PP, P, ctypes.POINTER(ctypes.c_uint32)]),
                "decode_attn_strerror": (ctypes.c_char_p, [I]),
                "decode_attn_max_partitions": (I, [PP]),
                "decode_attn_encode_fp8": (I, [P, ctypes.c_int64, P, P, P]),
                "decode_attn_encode_cb4": (I, [P, ctypes.c_int64, ctypes.c_int32, P, P, P, P, P]),
                "decode_attn_encode_codebook": (I, [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P, P, P,
                                                    P]),
                "decode_attn_codebook_lloyd_max": (I, [ctypes.c_int32, ctypes.c_double, P]),
                "decode_attn_debug_partition_bounds": (I, [P, P, PP, P]),
                "decode_attn_debug_dequant_blocks": (I, [P, P, P, P, ctypes.c_int32, ctypes.c_int32, P, PP, P]),
            }
            for name, (res, args) in sigs.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


def library():
    """The loaded ctypes CDLL (loads it on first use)."""
    return _load()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, what: str):
    if rc != DA_OK:
        raise DecodeAttnError(rc, what)


def decode_attn_strerror(status: int) -> str:
    return _load().decode_attn_strerror(int(status)).decode()


def decode_attn_workspace_bytes(params: da_params) -> int:
    return int(_load().decode_attn_workspace_bytes(ctypes.byref(params)))


def decode_attn_workspace_init(params: da_params, stream=None) -> None:
    _check(_load().decode_attn_workspace_init(ctypes.byref(params), _stream(stream)), "decode_attn_workspace_init")


def decode_attn_max_partitions(params: da_params) -> int:
    rc = _load().decode_attn_max_partitions(ctypes.byref(params))
    _check(min(rc, 0), "decode_attn_max_partitions")
    return int(rc)


def _call(name, q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables, context_lens, out,
          params, stream):
    fn = getattr(_load(), name)
    rc = fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales), _ptr(codebook),
            _ptr(sign_pattern), _ptr(block_tables), _ptr(context_lens), _ptr(out), ctypes.byref(params),
            _stream(stream))
    _check(rc, name)


def decode_attn_paged(q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables, context_lens,
                      out, params, stream=None) -> None:
    _call("decode_attn_paged", q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
          context_lens, out, params, stream)


def decode_attn_paged_static_workspace(q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern,
                                      block_tables, context_lens, out, params, stream=None) -> None:
    """decode_attn_paged for callers that cannot allocate device memory: the workspace is the
    library's own fixed 64 MiB device array (params.workspace is ignored). Calls that overlap
    on the GPU share that array and race; serialise them."""
    _call("decode_attn_paged_static_workspace", q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern,
          block_tables, context_lens, out, params, stream)


def decode_attn_rotate_q(q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                         context_lens, out, params, stream=None) -> None:
    _call("decode_attn_rotate_q", q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
          context_lens, out, params, stream)


def decode_attn_partition(q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                          context_lens, out, params, stream=None) -> None:
    _call("decode_attn_partition", q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
          context_lens, out, params, stream)


def decode_attn_reduce(q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables, context_lens,
                       out, params, stream=None) -> None:
    _call("decode_attn_reduce", q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
          context_lens, out, params, stream)


def decode_attn_get_device_error(params: da_params, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(_load().decode_attn_get_device_error(ctypes.byref(params), _stream(stream), ctypes.byref(v)),
           "decode_attn_get_device_error")
    return int(v.value)


def decode_attn_encode_fp8(x, n, codes, scale_out, stream=None) -> None:
    _check(_load().decode_attn_encode_fp8(_ptr(x), int(n), _ptr(codes), _ptr(scale_out), _stream(stream)),
           "decode_attn_encode_fp8")


def decode_attn_encode_cb4(x, num_vectors, head_dim, sign_pattern, codebook, packed, scales, stream=None) -> None:
    _check(_load().decode_attn_encode_cb4(_ptr(x), int(num_vectors), int(head_dim), _ptr(sign_pattern),
                                          _ptr(codebook), _ptr(packed), _ptr(scales), _stream(stream)),
           "decode_attn_encode_cb4")


def decode_attn_encode_codebook(x, num_vectors, head_dim, bits, sign_pattern, codebook, packed, scales,
                                stream=None) -> None:
    _check(_load().decode_attn_encode_codebook(_ptr(x), int(num_vectors), int(head_dim), int(bits),
                                               _ptr(sign_pattern), _ptr(codebook), _ptr(packed), _ptr(scales),
                                               _stream(stream)), "decode_attn_encode_codebook")


def decode_attn_codebook_lloyd_max(levels: int, sigma: float):
    """Host call: the Lloyd-Max codebook as a list of `levels` floats (ascending)."""
    buf = (ctypes.c_float * int(levels))()
    _check(_load().decode_attn_codebook_lloyd_max(int(levels), float(sigma), buf), "decode_attn_codebook_lloyd_max")
    return [float(v) for v in buf]


def decode_attn_debug_partition_bounds(context_lens, bounds, params: da_params, stream=None) -> None:
    _check(_load().decode_attn_debug_partition_bounds(_ptr(context_lens), _ptr(bounds), ctypes.byref(params),
                                                      _stream(stream)), "decode_attn_debug_partition_bounds")


def decode_attn_debug_dequant_blocks(cache, scales, codebook, block_ids, n, which, out, params: da_params,
                                     stream=None) -> None:
    _check(_load().decode_attn_debug_dequant_blocks(_ptr(cache), _ptr(scales), _ptr(codebook), _ptr(block_ids),
                                                    int(n), int(which), _ptr(out), ctypes.byref(params),
                                                    _stream(stream)), "decode_attn_debug_dequant_blocks")
