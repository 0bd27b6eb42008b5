"""fp64 CPU oracle for single-token paged GQA decode attention and its KV encodings.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The product (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product: the two
share no code. The arithmetic lives in ``oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

What each function follows is cited beside it in ``oracle.c``:
  - attention.rs README, "KV Cache Formats" table and the split-K sentence under it;
  - turboquant-rs 0.4.1, src/cache/cuda/attention.rs, fused_attention().

Every function here is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

FMT = {"bf16": 0, "fp8": 1, "cb4": 2, "fp8k_cb4v": 3, "cb3k_cb4v": 4}
# (K side, V side) storage of each format
SIDES = {"bf16": ("bf16", "bf16"), "fp8": ("fp8", "fp8"), "cb4": ("cb4", "cb4"), "fp8k_cb4v": ("fp8", "cb4"),
         "cb3k_cb4v": ("cb3", "cb4")}
ERRORS = {0: "ok", -1: "invalid argument", -2: "block-table entry out of range", -3: "out of memory"}

_lib = None
_lock = threading.Lock()


def compile_source(src: str, out: str) -> str:
    """gcc -O2 without FMA contraction or fast-math; used for oracle.c (and, by the mutation
    test, for deliberately broken copies of it)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


@contextlib.contextmanager
def library_override(path: str):
    """Run the oracle's Python functions against another build of oracle.c (tests only)."""
    global _lib
    with _lock:
        saved = _lib
        _lib = _open(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build())
        return _lib


def _open(path: str):
    lib = ctypes.CDLL(path)
    P, I, I64, D, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
    sig = {
        "or_bf16_decode": (D, [ctypes.c_uint16]),
        "or_e4m3_decode": (D, [ctypes.c_uint8]),
        "or_e4m3_encode": (ctypes.c_uint8, [F]),
        "or_e4m3_decode_array": (None, [P, I64, P]),
        "or_e4m3_encode_array": (None, [P, I64, P]),
        "or_fp8_quantize": (F, [P, I64, P, I]),
        "or_hadamard": (None, [I, P]),
        "or_lloyd_max": (I, [I, D, D, I, P, P]),
        "or_cb_nearest": (I, [D, P, I]),
        "or_cb4_encode": (I, [P, I64, I, P, P, P, P, I]),
        "or_cb4_dequant_rotated": (None, [P, P, I64, I, P, P]),
        "or_cb4_dequant": (None, [P, P, I64, I, P, P, P]),
        "or_cb_encode": (I, [I, P, I64, I, P, P, P, P, I]),
        "or_cb_dequant_rotated": (None, [I, P, P, I64, I, P, P]),
        "or_cb_dequant": (None, [I, P, P, I64, I, P, P, P]),
        "or_partition_bounds": (I, [I, I, I, I, P, P, I]),
        "or_partition_bounds_multi": (I, [I, I, I, I, I, P, P, I]),
        "or_default_threads": (I, []),
        "or_decode_attention": (I, [I, I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, D, D, P, I, I, I, P, P,
                                    I, ctypes.POINTER(ctypes.c_int)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return int(_load().or_default_threads())


# ---------------------------------------------------------------- element formats
def bf16_decode(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64 values (the upper half of a binary32)."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.or_bf16_decode(int(x)) for x in b.ravel()], dtype=np.float64).reshape(b.shape)


def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().or_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even E4M3 codes of binary32 values, saturating at +-448."""
    a = _c(x, np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    _load().or_e4m3_encode_array(_ptr(a), a.size, _ptr(out))
    return out


def fp8_quantize(x, threads: int = 0):
    """One scale for the whole tensor: scale = amax / 448 (binary32), codes = E4M3(x / scale)."""
    a = _c(x, np.float32)
    codes = np.empty(a.shape, dtype=np.uint8)
    scale = _load().or_fp8_quantize(_ptr(a), a.size, _ptr(codes), threads)
    return codes, np.float32(scale)


# ---------------------------------------------------------------- Hadamard + codebook
def hadamard(D: int) -> np.ndarray:
    H = np.empty((D, D), dtype=np.float64)
    _load().or_hadamard(D, _ptr(H))
    return H


def lloyd_max(levels: int = 16, sigma: float = 1.0 / np.sqrt(128.0), tol: float = 1e-14, max_iter: int = 1_000_000):
    """Lloyd-Max levels for N(0, sigma^2): (fp64 levels, fp32 codebook, iterations)."""
    lv = np.empty(levels, dtype=np.float64)
    cb = np.empty(levels, dtype=np.float32)
    it = _load().or_lloyd_max(levels, float(sigma), float(tol), max_iter, _ptr(lv), _ptr(cb))
    if it < 0:
        raise RuntimeError("Lloyd-Max iteration did not converge")
    return lv, cb, int(it)


def cb_nearest(u: float, codebook) -> int:
    cb = _c(codebook, np.float32)
    return int(_load().or_cb_nearest(float(u), _ptr(cb), cb.size))


def cb4_encode(x, sign, codebook, threads: int = 0):
    """Encode vectors x[..., D] -> (packed uint8 [..., D/2], scales fp32 [...])."""
    a = _c(x, np.float32)
    D = a.shape[-1]
    nvec = a.size // D
    packed = np.empty(a.shape[:-1] + (D // 2,), dtype=np.uint8)
    scales = np.empty(a.shape[:-1], dtype=np.float32)
    rc = _load().or_cb4_encode(_ptr(a), nvec, D, _ptr(_c(sign, np.float32)), _ptr(_c(codebook, np.float32)),
                               _ptr(packed), _ptr(scales), threads)
    if rc:
        raise ValueError(ERRORS.get(rc, rc))
    return packed, scales


def cb_encode(bits, x, sign, codebook, threads: int = 0):
    """b-bit codebook encoding of vectors x[..., D] -> (packed uint8 [..., D*bits/8], scales fp32)."""
    a = _c(x, np.float32)
    D = a.shape[-1]
    nvec = a.size // D
    packed = np.empty(a.shape[:-1] + (D * bits // 8,), dtype=np.uint8)
    scales = np.empty(a.shape[:-1], dtype=np.float32)
    rc = _load().or_cb_encode(int(bits), _ptr(a), nvec, D, _ptr(_c(sign, np.float32)),
                              _ptr(_c(codebook, np.float32)), _ptr(packed), _ptr(scales), threads)
    if rc:
        raise ValueError(ERRORS.get(rc, rc))
    return packed, scales


def cb_dequant_rotated(bits, packed, scales, codebook) -> np.ndarray:
    p = _c(packed, np.uint8)
    s = _c(scales, np.float32)
    D = p.shape[-1] * 8 // bits
    out = np.empty(p.shape[:-1] + (D,), dtype=np.float64)
    _load().or_cb_dequant_rotated(int(bits), _ptr(p), _ptr(s), s.size, D, _ptr(_c(codebook, np.float32)), _ptr(out))
    return out


def cb_dequant(bits, packed, scales, codebook, sign) -> np.ndarray:
    p = _c(packed, np.uint8)
    s = _c(scales, np.float32)
    D = p.shape[-1] * 8 // bits
    out = np.empty(p.shape[:-1] + (D,), dtype=np.float64)
    _load().or_cb_dequant(int(bits), _ptr(p), _ptr(s), s.size, D, _ptr(_c(codebook, np.float32)),
                          _ptr(_c(sign, np.float32)), _ptr(out))
    return out


def cb4_dequant_rotated(packed, scales, codebook) -> np.ndarray:
    """scale * codebook[idx] per coordinate, in the rotated basis (fp64)."""
    p = _c(packed, np.uint8)
    s = _c(scales, np.float32)
    D = p.shape[-1] * 2
    out = np.empty(p.shape[:-1] + (D,), dtype=np.float64)
    _load().or_cb4_dequant_rotated(_ptr(p), _ptr(s), s.size, D, _ptr(_c(codebook, np.float32)), _ptr(out))
    return out


def cb4_dequant(packed, scales, codebook, sign) -> np.ndarray:
    """Dequantise back to the original basis: diag(sign) H (scale * cb[idx]) / sqrt(D)."""
    p = _c(packed, np.uint8)
    s = _c(scales, np.float32)
    D = p.shape[-1] * 2
    out = np.empty(p.shape[:-1] + (D,), dtype=np.float64)
    _load().or_cb4_dequant(_ptr(p), _ptr(s), s.size, D, _ptr(_c(codebook, np.float32)), _ptr(_c(sign, np.float32)),
                           _ptr(out))
    return out


# ---------------------------------------------------------------- attention
def partition_bounds(L: int, window: int = 0, partition_size: int = 512, split_threshold: int = 1024,
                     query_len: int = 1):
    """[(start, end), ...] of the partitions of one sequence of length L with query_len
    query tokens (the last query_len positions)."""
    cap = 1 << 16
    st = np.empty(cap, dtype=np.int32)
    en = np.empty(cap, dtype=np.int32)
    if query_len == 1:
        n = _load().or_partition_bounds(int(L), int(window), int(partition_size), int(split_threshold), _ptr(st),
                                        _ptr(en), cap)
    else:
        n = _load().or_partition_bounds_multi(int(L), int(query_len), int(window), int(partition_size),
                                              int(split_threshold), _ptr(st), _ptr(en), cap)
    return [(int(st[i]), int(en[i])) for i in range(n)]


def decode_attention(q_bits, k_cache, v_cache, block_tables, context_lens, *, kv_format: str, num_kv_heads: int,
                     softmax_scale: float, softcap: float = 0.0, window: int = 0, partition_size: int = 0,
                     split_threshold: int = 1024, k_scales=None, v_scales=None, codebook=None, sign_pattern=None,
                     alibi_slopes=None, select=None, threads: int = 0, return_threads: bool = False):
    """fp64 paged GQA decode attention.

    q_bits: uint16 bf16 bit patterns [B, Hq, D], or [B, T, Hq, D] for T query tokens per
    sequence (positions L-T .. L-1, causal). Caches: [num_blocks, Hkv, bs, D] uint16
    (bf16 bits) or uint8 (E4M3 codes), or [num_blocks, Hkv, bs, D/2] uint8 (packed 4-bit).
    k_scales/v_scales: fp8 -> one value each; cb4 -> [num_blocks, Hkv, bs] fp32.
    alibi_slopes: optional [Hq] slopes; the score of key position t for a query at position
    pos gets slope_h * (t - pos) added after scaling and softcap.
    select: optional list of (b, h) (or (b, j, h) with T query tokens); then the result is
    [len(select), D] in that order, else [B, Hq, D] (or [B, T, Hq, D]). partition_size 0
    computes without partitions.
    """
    q = _c(q_bits, np.uint16)
    multi = q.ndim == 4
    if not multi:
        q = q[:, None]
    B, T, Hq, D = q.shape
    kf = FMT[kv_format]
    kc = _c(k_cache, np.uint16 if kf == 0 else np.uint8)
    vc = _c(v_cache, np.uint16 if kf == 0 else np.uint8)
    if k_scales is not None and SIDES[kv_format][0] == "fp8":
        k_scales = np.atleast_1d(k_scales)
    num_blocks, hkv, bs = kc.shape[:3]
    if hkv != num_kv_heads:
        raise ValueError("cache head count does not match num_kv_heads")
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    ks = _c(np.atleast_1d(k_scales), np.float32) if k_scales is not None else None
    vs = _c(np.atleast_1d(v_scales), np.float32) if v_scales is not None else None
    if select is None:
        rows = None
        out = np.zeros((B, T, Hq, D), dtype=np.float64)
    else:
        rows = np.full(B * T * Hq, -1, dtype=np.int32)
        for i, key in enumerate(select):
            b, jq, h = key if len(key) == 3 else (key[0], 0, key[1])
            r = (b * T + jq) * Hq + h
            if rows[r] >= 0:
                raise ValueError("duplicate entry in select")
            rows[r] = i
        out = np.zeros((len(select), D), dtype=np.float64)
    slopes = None
    if alibi_slopes is not None:
        slopes = _c(alibi_slopes, np.float32)
        if slopes.shape != (Hq,):
            raise ValueError("alibi_slopes must hold one slope per query head")
    used = ctypes.c_int(0)
    rc = _load().or_decode_attention(
        B, T, Hq, num_kv_heads, D, bs, kf, num_blocks, bt.shape[1], _ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
        _ptr(_c(codebook, np.float32)), _ptr(_c(sign_pattern, np.float32)), _ptr(bt), _ptr(cl),
        float(softmax_scale), float(softcap), _ptr(slopes), int(window), int(partition_size), int(split_threshold),
        _ptr(rows), _ptr(out), int(threads), ctypes.byref(used))
    if rc:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")
    if select is None and not multi:
        out = out[:, 0]
    return (out, used.value) if return_threads else out
