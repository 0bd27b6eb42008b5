"""Single-token paged GQA decode attention for GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind a C-ABI shared library
(include/decode_attn.h, built from csrc/ by ``build.build()``); this package is its
ctypes binding (``_binding``) plus the seeded synthetic input generators (``workloads``).
"""
from ._binding import (  # noqa: F401
    DA_DEVERR_BLOCK_ID,
    DA_DEVERR_CONTEXT_LEN,
    DA_DEVERR_SMEM_LAYOUT,
    DA_DEVERR_TIMEOUT,
    DA_KV_BF16,
    DA_KV_CB3K_CB4V,
    DA_KV_CB4,
    DA_KV_FP8_E4M3,
    DA_KV_FP8K_CB4V,
    KV_FORMATS,
    LIB_PATH,
    DecodeAttnError,
    attach_workspace,
    da_params,
    decode_attn_debug_dequant_blocks,
    decode_attn_codebook_lloyd_max,
    decode_attn_debug_partition_bounds,
    decode_attn_encode_cb4,
    decode_attn_encode_codebook,
    decode_attn_encode_fp8,
    decode_attn_get_device_error,
    decode_attn_max_partitions,
    decode_attn_paged,
    decode_attn_paged_static_workspace,
    decode_attn_partition,
    decode_attn_reduce,
    decode_attn_rotate_q,
    decode_attn_strerror,
    decode_attn_workspace_bytes,
    decode_attn_workspace_init,
    library,
    make_params,
)
