"""CPU oracle for the FP8 paged KV-cache path -- TEST INFRASTRUCTURE.

Plain, slow, single-threaded C (``fp8kv_oracle.c``) behind numpy-facing
wrappers.  Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU
baseline leg may import this package; the product library never does.  It
shares no code with the CUDA path.

Arrays: bf16 tensors travel as ``np.uint16`` bit patterns, caches as raw bytes
(``np.uint8``; a bf16 cache is a ``np.uint16`` array), indices as int32/int64.
"""
import ctypes
import numpy as np

from . import build as _build

_lib = None

E4M3, BF16 = 0, 1


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(_build.build())
        _declare(_lib)
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def _declare(L):
    vp, i32, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                             ctypes.c_double, ctypes.c_size_t)
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [f32]
    L.oracle_e4m3_decode.restype = f64
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_encode_array.argtypes = [vp, sz, vp]
    L.oracle_e4m3_decode_array.argtypes = [vp, sz, vp]
    L.oracle_e4m3_encode_bits_range.argtypes = [ctypes.c_uint32, sz, vp]
    L.oracle_cache_insert.restype = i32
    L.oracle_cache_insert.argtypes = [vp, vp, vp, i32, i32, i32, f32, f32, vp, vp, i32, i32, i32]
    L.oracle_cache_insert_per_head.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32, i32]
    L.oracle_paged_attention_per_head.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                                  vp, vp, f64, i32, vp]
    L.oracle_rope_table.argtypes = [f64, i32, i32, vp]
    L.oracle_norm_rope_row.restype = i32
    L.oracle_norm_rope_row.argtypes = [vp, vp, f32, vp, i32, vp]
    L.oracle_qk_norm_rope_insert.restype = i32
    L.oracle_qk_norm_rope_insert.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, i32, vp, vp,
                                             i32, i32, i32, i32, f32, f32, vp, vp, i32, i32]
    attn = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, f64, f64, f64, i32]
    L.oracle_paged_attention.restype = i32
    L.oracle_paged_attention.argtypes = attn + [vp]
    L.oracle_paged_attention_rows.restype = i32
    L.oracle_paged_attention_rows.argtypes = attn + [vp, i32, vp]
    L.oracle_paged_attention_split_rows.restype = i32
    L.oracle_paged_attention_split_rows.argtypes = attn + [i32, vp, i32, vp]


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ codec

def e4m3_encode(x):
    """fp32 array -> E4M3FN codes (uint8), saturating RNE."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_encode_bits(first, n):
    """Codes of the fp32 bit patterns first .. first+n-1."""
    out = np.empty(n, np.uint8)
    lib().oracle_e4m3_encode_bits_range(first, n, _p(out))
    return out


def e4m3_decode(c):
    """E4M3FN codes -> float64 values (NaN for S.1111.111)."""
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().oracle_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


# ----------------------------------------------------------------- insert

def cache_insert(k, v, slot_mapping, k_scale, v_scale, k_cache, v_cache, cache_dtype=E4M3):
    """Insert bf16 K/V rows ``[T][Hkv][D]`` into the caches in place.

    Caches are ``[num_pages][Hkv][page_size][D]`` (uint8 for E4M3, uint16 for bf16).
    """
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    T, Hkv, D = k.shape
    num_pages, _, page_size, _ = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    rc = lib().oracle_cache_insert(_p(k), _p(v), _p(slot_mapping), T, Hkv, D,
                                   float(k_scale), float(v_scale), _p(k_cache), _p(v_cache),
                                   num_pages, page_size, cache_dtype)
    if rc:
        raise ValueError("oracle_cache_insert: bad arguments")


def cache_insert_per_head(k, v, slot_mapping, k_scales, v_scales, k_cache, v_cache):
    """Insert bf16 K/V rows ``[T][Hkv][D]`` into E4M3 caches in place, head h
    encoded with its own scale k_scales[h] (v_scales[h]), fp32."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    T, Hkv, D = k.shape
    ks = _c(np.asarray(k_scales, np.float32).reshape(-1), np.float32)
    vs = _c(np.asarray(v_scales, np.float32).reshape(-1), np.float32)
    if ks.shape[0] != Hkv or vs.shape[0] != Hkv:
        raise ValueError("one scale per KV head")
    num_pages, _, page_size, _ = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous and k_cache.dtype == np.uint8
    rc = lib().oracle_cache_insert_per_head(_p(k), _p(v), _p(slot_mapping), T, Hkv, D, _p(ks), _p(vs),
                                            _p(k_cache), _p(v_cache), num_pages, page_size)
    if rc:
        raise ValueError("oracle_cache_insert_per_head: bad arguments")


# ------------------------------------------------------- RMSNorm and RoPE

def rope_table(theta, max_pos, D):
    """fp32 ``[max_pos][D]``: cos of the D/2 frequencies, then their sines."""
    out = np.empty((max_pos, D), np.float32)
    lib().oracle_rope_table(float(theta), max_pos, D, _p(out))
    return out


def norm_rope_row(x, w, eps, cs_row):
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    cs_row = _c(cs_row, np.float32)
    out = np.empty(x.shape, np.uint16)
    rc = lib().oracle_norm_rope_row(_p(x), _p(w), float(eps), _p(cs_row), x.shape[-1], _p(out))
    if rc:
        raise ValueError("oracle_norm_rope_row: bad arguments")
    return out


def qk_norm_rope_insert(q, k, v, positions, q_norm_w, k_norm_w, eps, cos_sin, slot_mapping,
                        k_scale, v_scale, k_cache, v_cache):
    """Returns q_out (bf16 bits) and inserts rotated K / raw V into the E4M3 caches."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    positions = _c(positions, np.int64)
    slot_mapping = _c(slot_mapping, np.int64)
    q_norm_w = _c(q_norm_w, np.uint16)
    k_norm_w = _c(k_norm_w, np.uint16)
    cos_sin = _c(cos_sin, np.float32)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    num_pages, _, page_size, _ = k_cache.shape
    q_out = np.empty_like(q)
    rc = lib().oracle_qk_norm_rope_insert(
        _p(q), _p(k), _p(v), _p(positions), _p(q_norm_w), _p(k_norm_w), float(eps),
        _p(cos_sin), cos_sin.shape[0], _p(q_out), _p(slot_mapping), T, Hq, Hkv, D,
        float(k_scale), float(v_scale), _p(k_cache), _p(v_cache), num_pages, page_size)
    if rc:
        raise ValueError("oracle_qk_norm_rope_insert: bad arguments")
    return q_out


# -------------------------------------------------------------- attention

def _attn_args(q, k_cache, v_cache, cache_dtype, block_table, seq_lens, k_scale, v_scale,
               sm_scale, window_left):
    q = _c(q, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, M, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    keep = (q, block_table, seq_lens)
    args = [_p(q), _p(k_cache), _p(v_cache), cache_dtype, _p(block_table), block_table.shape[1],
            _p(seq_lens), B, M, Hq, Hkv, D, page_size, num_pages, float(k_scale),
            float(v_scale), float(sm_scale), int(window_left)]
    return args, keep, (B, M, Hq, D)


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, sm_scale,
                    window_left=-1, cache_dtype=E4M3):
    """float64 ``[B][M][Hq][D]``: softmax(Q Kd^T * sm_scale + mask) Vd."""
    args, keep, (B, M, Hq, D) = _attn_args(q, k_cache, v_cache, cache_dtype, block_table,
                                           seq_lens, k_scale, v_scale, sm_scale, window_left)
    out = np.empty((B, M, Hq, D), np.float64)
    if lib().oracle_paged_attention(*args, _p(out)):
        raise ValueError("oracle_paged_attention: bad arguments")
    return out


def paged_attention_rows(q, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, sm_scale,
                         rows, window_left=-1, cache_dtype=E4M3, split_tokens=0):
    """float64 ``[n][D]`` for rows ``[(b, m, h), ...]``; split_tokens > 0 uses the
    partition + log-sum-exp combine instead of one softmax."""
    args, keep, (B, M, Hq, D) = _attn_args(q, k_cache, v_cache, cache_dtype, block_table,
                                           seq_lens, k_scale, v_scale, sm_scale, window_left)
    rows = _c(rows, np.int32).reshape(-1, 3)
    out = np.empty((rows.shape[0], D), np.float64)
    if split_tokens > 0:
        rc = lib().oracle_paged_attention_split_rows(*args, int(split_tokens), _p(rows),
                                                     rows.shape[0], _p(out))
    else:
        rc = lib().oracle_paged_attention_rows(*args, _p(rows), rows.shape[0], _p(out))
    if rc:
        raise ValueError("oracle_paged_attention_rows: bad arguments")
    return out


def paged_attention_per_head(q, k_cache, v_cache, block_table, seq_lens, k_scales, v_scales, sm_scale,
                             window_left=-1):
    """float64 ``[B][M][Hq][D]`` over an E4M3 cache whose KV head hk is
    dequantized with k_scales[hk], v_scales[hk]."""
    q = _c(q, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, M, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_cache.shape
    ks = _c(np.asarray(k_scales, np.float64).reshape(-1), np.float64)
    vs = _c(np.asarray(v_scales, np.float64).reshape(-1), np.float64)
    if ks.shape[0] != Hkv or vs.shape[0] != Hkv:
        raise ValueError("one scale per KV head")
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous and k_cache.dtype == np.uint8
    out = np.empty((B, M, Hq, D), np.float64)
    rc = lib().oracle_paged_attention_per_head(_p(q), _p(k_cache), _p(v_cache), _p(block_table),
                                               block_table.shape[1], _p(seq_lens), B, M, Hq, Hkv, D,
                                               page_size, num_pages, _p(ks), _p(vs), float(sm_scale),
                                               int(window_left), _p(out))
    if rc:
        raise ValueError("oracle_paged_attention_per_head: bad arguments")
    return out
