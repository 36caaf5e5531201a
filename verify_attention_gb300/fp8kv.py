"""Thin ctypes binding of libfp8kv.so (include/fp8kv.h), same names as the C ABI.

Only argument marshalling happens here: tensors become device pointers and
sizes, the current torch stream becomes the cudaStream_t, and a non-zero
status raises ``Fp8kvError``.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback: if the library is missing, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp8kv.so")

FP8KV_CACHE_E4M3 = 0
FP8KV_CACHE_BF16 = 1
DEV_BAD_SLOT, DEV_BAD_POSITION, DEV_BAD_SEQ_LEN, DEV_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8

_lib = None


class Fp8kvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status} ({fp8kv_status_string(status)})")


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m verify_attention_gb300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_float,
                                 ctypes.c_size_t)
        L.fp8kv_cache_insert.restype = i32
        L.fp8kv_cache_insert.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32, i32, i32, vp]
        L.fp8kv_qk_norm_rope_insert.restype = i32
        L.fp8kv_qk_norm_rope_insert.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, i32, vp, vp, i32, i32,
                                                i32, i32, vp, vp, vp, vp, i32, i32, vp]
        L.fp8kv_paged_attention_plan.restype = i32
        L.fp8kv_paged_attention_plan.argtypes = [i32] * 9 + [ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.fp8kv_paged_attention_workspace_size.restype = sz
        L.fp8kv_paged_attention_workspace_size.argtypes = [i32] * 9
        L.fp8kv_paged_attention.restype = i32
        L.fp8kv_paged_attention.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32,
                                            i32, i32, vp, vp, f32, i32, i32, vp, sz, vp, vp]
        L.fp8kv_append_paged_attention.restype = i32
        L.fp8kv_append_paged_attention.argtypes = [vp, vp] + L.fp8kv_paged_attention.argtypes
        L.fp8kv_cache_insert_per_head.restype = i32
        L.fp8kv_cache_insert_per_head.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32, i32, vp]
        L.fp8kv_paged_attention_per_head.restype = i32
        L.fp8kv_paged_attention_per_head.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32,
                                                     i32, i32, vp, vp, f32, i32, i32, vp, sz, vp, vp]
        L.fp8kv_append_paged_attention_per_head.restype = i32
        L.fp8kv_append_paged_attention_per_head.argtypes = [vp, vp] + L.fp8kv_paged_attention_per_head.argtypes
        L.fp8kv_paged_attention_noalloc.restype = i32
        L.fp8kv_paged_attention_noalloc.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                                                    i32, i32, i32, vp, vp, f32, i32, i32, vp, vp]
        L.fp8kv_paged_attention_layers_workspace_size.restype = sz
        L.fp8kv_paged_attention_layers_workspace_size.argtypes = [i32] * 5
        L.fp8kv_paged_attention_layers.restype = i32
        L.fp8kv_paged_attention_layers.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, sz, vp]
        L.fp8kv_e4m3_encode_bits.restype = i32
        L.fp8kv_e4m3_encode_bits.argtypes = [u32, sz, vp, vp]
        L.fp8kv_selftest_bounded_wait.restype = i32
        L.fp8kv_selftest_bounded_wait.argtypes = [ctypes.c_uint, vp]
        L.fp8kv_status_string.restype = ctypes.c_char_p
        L.fp8kv_status_string.argtypes = [i32]
        L.fp8kv_last_dispatch.restype = i32
        L.fp8kv_last_dispatch.argtypes = [ctypes.c_char_p, sz]
        L.fp8kv_launch_count.restype = ctypes.c_ulonglong
        L.fp8kv_launch_count.argtypes = []
        L.fp8kv_device_status.restype = i32
        L.fp8kv_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]) -> int:
    # plain ints: ctypes converts them for c_void_p arguments without a wrapper object
    return t.data_ptr() if t is not None else 0


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn, rc):
    if rc != 0:
        raise Fp8kvError(fn, rc)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _cache_dtype(cache: torch.Tensor) -> int:
    if cache.dtype == torch.uint8:
        return FP8KV_CACHE_E4M3
    if cache.dtype == torch.bfloat16:
        return FP8KV_CACHE_BF16
    raise ValueError("cache must be uint8 (E4M3 codes) or bfloat16")


def fp8kv_status_string(status: int) -> str:
    return lib().fp8kv_status_string(status).decode()


def fp8kv_cache_insert(k, v, slot_mapping, k_scale, v_scale, k_cache, v_cache, stream=None):
    """k, v bf16 [T][Hkv][D]; slot_mapping int64 [T]; scales fp32 [1] (E4M3 only);
    caches [num_pages][Hkv][page_size][D] uint8 (E4M3) or bf16."""
    dt = _cache_dtype(k_cache)
    _dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16)
    _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache")
    T, Hkv, D = k.shape
    num_pages, _, page_size, _ = k_cache.shape
    rc = lib().fp8kv_cache_insert(_ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, D, _ptr(k_scale),
                                  _ptr(v_scale), _ptr(k_cache), _ptr(v_cache), num_pages, page_size,
                                  dt, _stream(stream))
    _check("fp8kv_cache_insert", rc)


def _head_scales(k_scale, v_scale, Hkv):
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _dev(t, n, torch.float32)
        if t.numel() != Hkv:
            raise ValueError(f"{n} must hold one fp32 scale per KV head ({Hkv}), got {t.numel()}")


def fp8kv_cache_insert_per_head(k, v, slot_mapping, k_scale, v_scale, k_cache, v_cache, stream=None):
    """fp8kv_cache_insert on an E4M3 cache with per-head scales fp32 [Hkv]."""
    _dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16)
    _dev(slot_mapping, "slot_mapping", torch.int64)
    _dev(k_cache, "k_cache", torch.uint8), _dev(v_cache, "v_cache", torch.uint8)
    T, Hkv, D = k.shape
    _head_scales(k_scale, v_scale, Hkv)
    num_pages, _, page_size, _ = k_cache.shape
    rc = lib().fp8kv_cache_insert_per_head(_ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, D, _ptr(k_scale),
                                           _ptr(v_scale), _ptr(k_cache), _ptr(v_cache), num_pages, page_size,
                                           _stream(stream))
    _check("fp8kv_cache_insert_per_head", rc)


def fp8kv_qk_norm_rope_insert(q, k, v, positions, q_norm_w, k_norm_w, eps, cos_sin, q_out,
                              slot_mapping, k_scale, v_scale, k_cache, v_cache, stream=None):
    """Fused Q/K RMSNorm + RoPE + E4M3 insert; writes q_out (bf16 [T][Hq][D])."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (q_out, "q_out"), (q_norm_w, "q_norm_w"),
                 (k_norm_w, "k_norm_w")):
        _dev(t, n, torch.bfloat16)
    _dev(positions, "positions", torch.int64), _dev(slot_mapping, "slot_mapping", torch.int64)
    _dev(cos_sin, "cos_sin", torch.float32), _dev(k_cache, "k_cache", torch.uint8)
    _dev(v_cache, "v_cache", torch.uint8)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    num_pages, _, page_size, _ = k_cache.shape
    rc = lib().fp8kv_qk_norm_rope_insert(
        _ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(q_norm_w), _ptr(k_norm_w), float(eps),
        _ptr(cos_sin), cos_sin.shape[0], _ptr(q_out), _ptr(slot_mapping), T, Hq, Hkv, D, _ptr(k_scale),
        _ptr(v_scale), _ptr(k_cache), _ptr(v_cache), num_pages, page_size, _stream(stream))
    _check("fp8kv_qk_norm_rope_insert", rc)


def fp8kv_paged_attention_plan(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left, split_tokens=0):
    ns, st = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().fp8kv_paged_attention_plan(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left,
                                          split_tokens, ctypes.byref(ns), ctypes.byref(st))
    _check("fp8kv_paged_attention_plan", rc)
    return ns.value, st.value


def fp8kv_paged_attention_workspace_size(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left,
                                         split_tokens=0) -> int:
    n = lib().fp8kv_paged_attention_workspace_size(B, M, Hq, Hkv, D, page_size, max_seq_len,
                                                   window_left, split_tokens)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("fp8kv_paged_attention_workspace_size: bad arguments")
    return n


def fp8kv_paged_attention(q, k_cache, v_cache, block_table, seq_lens, max_seq_len, k_scale, v_scale,
                          sm_scale, window_left=-1, split_tokens=0, workspace=None, out=None,
                          num_pages=None, stream=None):
    """q bf16 [B][M][Hq][D]; caches [num_pages][Hkv][page_size][D]; block_table int32
    [B][max_pages_per_seq]; seq_lens int32 [B] (context incl. the M new rows).
    Returns out bf16 [B][M][Hq][D].  ``workspace`` (uint8 CUDA tensor) is
    allocated by torch here when not given and needed."""
    dt = _cache_dtype(k_cache)
    _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache")
    _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32)
    B, M, Hq, D = q.shape
    P, Hkv, page_size, _ = k_cache.shape
    if num_pages is None:
        num_pages = P
    need = fp8kv_paged_attention_workspace_size(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left,
                                                split_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    rc = lib().fp8kv_paged_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), int(max_seq_len), B, M, Hq, Hkv, D, page_size, int(num_pages), _ptr(k_scale),
        _ptr(v_scale), float(sm_scale), int(window_left), int(split_tokens), _ptr(workspace),
        workspace.numel() if workspace is not None else 0, _ptr(out), _stream(stream))
    _check("fp8kv_paged_attention", rc)
    return out


def fp8kv_append_paged_attention(k_new, v_new, q, k_cache, v_cache, block_table, seq_lens, max_seq_len, k_scale,
                                 v_scale, sm_scale, window_left=-1, split_tokens=0, workspace=None, out=None,
                                 num_pages=None, stream=None):
    """fp8kv_paged_attention after writing the M new tokens of each sequence
    (k_new, v_new bf16 [B][M][Hkv][D]) to the cache at positions L - M + m."""
    dt = _cache_dtype(k_cache)
    _dev(k_new, "k_new", torch.bfloat16), _dev(v_new, "v_new", torch.bfloat16)
    _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache")
    _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32)
    B, M, Hq, D = q.shape
    P, Hkv, page_size, _ = k_cache.shape
    if tuple(k_new.shape) != (B, M, Hkv, D) or tuple(v_new.shape) != (B, M, Hkv, D):
        raise ValueError("k_new, v_new must be [B][M][Hkv][D]")
    if num_pages is None:
        num_pages = P
    need = fp8kv_paged_attention_workspace_size(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left,
                                                split_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    rc = lib().fp8kv_append_paged_attention(
        _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), int(max_seq_len), B, M, Hq, Hkv, D, page_size, int(num_pages),
        _ptr(k_scale), _ptr(v_scale), float(sm_scale), int(window_left), int(split_tokens), _ptr(workspace),
        workspace.numel() if workspace is not None else 0, _ptr(out), _stream(stream))
    _check("fp8kv_append_paged_attention", rc)
    return out


def fp8kv_paged_attention_per_head(q, k_cache, v_cache, block_table, seq_lens, max_seq_len, k_scale, v_scale,
                                   sm_scale, window_left=-1, split_tokens=0, workspace=None, out=None,
                                   num_pages=None, k_new=None, v_new=None, stream=None):
    """fp8kv_paged_attention on an E4M3 cache with per-head scales fp32 [Hkv];
    with k_new, v_new (bf16 [B][M][Hkv][D]) the append variant
    (fp8kv_append_paged_attention_per_head)."""
    _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache", torch.uint8), _dev(v_cache, "v_cache", torch.uint8)
    _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32)
    B, M, Hq, D = q.shape
    P, Hkv, page_size, _ = k_cache.shape
    _head_scales(k_scale, v_scale, Hkv)
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        _dev(k_new, "k_new", torch.bfloat16), _dev(v_new, "v_new", torch.bfloat16)
        if tuple(k_new.shape) != (B, M, Hkv, D) or tuple(v_new.shape) != (B, M, Hkv, D):
            raise ValueError("k_new, v_new must be [B][M][Hkv][D]")
    if num_pages is None:
        num_pages = P
    need = fp8kv_paged_attention_workspace_size(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left,
                                                split_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
            int(max_seq_len), B, M, Hq, Hkv, D, page_size, int(num_pages), _ptr(k_scale), _ptr(v_scale),
            float(sm_scale), int(window_left), int(split_tokens), _ptr(workspace),
            workspace.numel() if workspace is not None else 0, _ptr(out), _stream(stream))
    if k_new is None:
        _check("fp8kv_paged_attention_per_head", lib().fp8kv_paged_attention_per_head(*args))
    else:
        _check("fp8kv_append_paged_attention_per_head",
               lib().fp8kv_append_paged_attention_per_head(_ptr(k_new), _ptr(v_new), *args))
    return out


def fp8kv_append_paged_attention_per_head(k_new, v_new, q, k_cache, v_cache, block_table, seq_lens, max_seq_len,
                                          k_scale, v_scale, sm_scale, window_left=-1, split_tokens=0,
                                          workspace=None, out=None, num_pages=None, stream=None):
    """fp8kv_append_paged_attention on an E4M3 cache with per-head scales fp32 [Hkv]."""
    if k_new is None or v_new is None:
        raise ValueError("k_new and v_new are required")
    return fp8kv_paged_attention_per_head(q, k_cache, v_cache, block_table, seq_lens, max_seq_len, k_scale, v_scale,
                                          sm_scale, window_left, split_tokens, workspace, out, num_pages, k_new,
                                          v_new, stream)


class PreparedAttention:
    """fp8kv_append_paged_attention (k_new, v_new given) or
    fp8kv_paged_attention over fixed tensors, marshalled once: each call
    passes the prepared arguments and the stream, nothing else.  For serving
    loops whose caches, metadata and buffers stay at fixed addresses; the
    tensors must outlive the object."""

    def __init__(self, q, k_cache, v_cache, block_table, seq_lens, max_seq_len, k_scale, v_scale, sm_scale,
                 window_left=-1, split_tokens=0, workspace=None, out=None, k_new=None, v_new=None, num_pages=None):
        dt = _cache_dtype(k_cache)
        _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache")
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32)
        B, M, Hq, D = q.shape
        P, Hkv, page_size, _ = k_cache.shape
        if (k_new is None) != (v_new is None):
            raise ValueError("k_new and v_new go together")
        if k_new is not None:
            for t, n in ((k_new, "k_new"), (v_new, "v_new")):
                _dev(t, n, torch.bfloat16)
                if tuple(t.shape) != (B, M, Hkv, D):
                    raise ValueError(f"{n} must be [B][M][Hkv][D]")
        need = fp8kv_paged_attention_workspace_size(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left,
                                                    split_tokens)
        if workspace is None and need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if out is None:
            out = torch.empty_like(q)
        if out.shape != q.shape:
            raise ValueError("out must have the shape of q")
        self.out, self._keep = out, (q, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, workspace, k_new,
                                     v_new)
        args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                int(max_seq_len), B, M, Hq, Hkv, D, page_size, int(P if num_pages is None else num_pages),
                _ptr(k_scale), _ptr(v_scale), float(sm_scale), int(window_left), int(split_tokens), _ptr(workspace),
                workspace.numel() if workspace is not None else 0, _ptr(out))
        if k_new is not None:
            self._fn, self._name = lib().fp8kv_append_paged_attention, "fp8kv_append_paged_attention"
            self._args = (_ptr(k_new), _ptr(v_new), *args)
        else:
            self._fn, self._name = lib().fp8kv_paged_attention, "fp8kv_paged_attention"
            self._args = args

    def __call__(self, stream=None):
        rc = self._fn(*self._args, _stream(stream))
        if rc:
            raise Fp8kvError(self._name, rc)
        return self.out


def fp8kv_paged_attention_noalloc(q, k_cache, v_cache, block_table, seq_lens, max_seq_len, k_scale, v_scale,
                                  sm_scale, out, window_left=-1, split_tokens=0, num_pages=None, stream=None):
    """fp8kv_paged_attention with the library's own fixed device workspace, for
    callers that cannot allocate device memory: ``out`` must be given, nothing
    is allocated here or in the library."""
    dt = _cache_dtype(k_cache)
    _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache")
    _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32)
    _dev(out, "out", torch.bfloat16)
    if out.shape != q.shape or out.device != q.device:
        raise ValueError(f"out must have the shape and device of q {tuple(q.shape)}, got {tuple(out.shape)}")
    B, M, Hq, D = q.shape
    P, Hkv, page_size, _ = k_cache.shape
    rc = lib().fp8kv_paged_attention_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        int(max_seq_len), B, M, Hq, Hkv, D, page_size, int(P if num_pages is None else num_pages),
        _ptr(k_scale), _ptr(v_scale), float(sm_scale), int(window_left), int(split_tokens), _ptr(out),
        _stream(stream))
    _check("fp8kv_paged_attention_noalloc", rc)
    return out


class fp8kv_layer(ctypes.Structure):
    """One layer of fp8kv_paged_attention_layers (include/fp8kv.h)."""
    _fields_ = [("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("max_pages_per_seq", ctypes.c_int), ("max_seq_len", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("window_left", ctypes.c_int), ("sm_scale", ctypes.c_float)]


def fp8kv_paged_attention_layers_workspace_size(n_layers, B, M, Hq, Hkv) -> int:
    n = lib().fp8kv_paged_attention_layers_workspace_size(n_layers, B, M, Hq, Hkv)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("fp8kv_paged_attention_layers_workspace_size: bad arguments")
    return n


class PagedAttentionLayers:
    """A prepared fp8kv_paged_attention_layers call over fixed tensors (the
    layers' persistent caches, metadata and buffers): the descriptors are
    marshalled once; each call passes them, the workspace and the stream.

    layers: dicts with q, k_new, v_new (or None), k_cache, v_cache,
    block_table, seq_lens, max_seq_len, k_scale, v_scale, sm_scale,
    window_left, out -- the arguments of fp8kv_append_paged_attention."""

    def __init__(self, layers, workspace=None):
        if not layers:
            raise ValueError("no layers")
        q0 = layers[0]["q"]
        B, M, Hq, D = q0.shape
        P0, Hkv, page_size, _ = layers[0]["k_cache"].shape
        self.shape = (B, M, Hq, Hkv, D, page_size)
        arr = (fp8kv_layer * len(layers))()
        self._keep = []
        for i, d in enumerate(layers):
            q, kc, vc = d["q"], d["k_cache"], d["v_cache"]
            _dev(q, "q", torch.bfloat16), _dev(kc, "k_cache", torch.uint8), _dev(vc, "v_cache", torch.uint8)
            _dev(d["block_table"], "block_table", torch.int32), _dev(d["seq_lens"], "seq_lens", torch.int32)
            _dev(d["out"], "out", torch.bfloat16)
            if tuple(q.shape) != (B, M, Hq, D) or tuple(d["out"].shape) != (B, M, Hq, D):
                raise ValueError(f"layer {i}: q and out must be {(B, M, Hq, D)}")
            if tuple(kc.shape[1:]) != (Hkv, page_size, D) or kc.shape != vc.shape:
                raise ValueError(f"layer {i}: caches must be [pages][{Hkv}][{page_size}][{D}]")
            kn, vn = d.get("k_new"), d.get("v_new")
            if (kn is None) != (vn is None):
                raise ValueError(f"layer {i}: k_new and v_new go together")
            if kn is not None:
                for t, n in ((kn, "k_new"), (vn, "v_new")):
                    _dev(t, n, torch.bfloat16)
                    if tuple(t.shape) != (B, M, Hkv, D):
                        raise ValueError(f"layer {i}: {n} must be {(B, M, Hkv, D)}")
            bt = d["block_table"]
            arr[i] = fp8kv_layer(_ptr(q), _ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(d["seq_lens"]),
                                 _ptr(d["k_scale"]), _ptr(d["v_scale"]), _ptr(d["out"]), bt.shape[1],
                                 int(d["max_seq_len"]), int(d.get("num_pages") or kc.shape[0]),
                                 int(d.get("window_left", -1)), float(d["sm_scale"]))
            self._keep.append(d)
        self.layers = arr
        self.n = len(layers)
        self.ws_bytes = fp8kv_paged_attention_layers_workspace_size(self.n, B, M, Hq, Hkv)
        if workspace is None:
            # the counters at its start must be zero before the first call
            workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=q0.device)
        self.workspace = workspace

    def __call__(self, stream=None):
        B, M, Hq, Hkv, D, page_size = self.shape
        rc = lib().fp8kv_paged_attention_layers(ctypes.byref(self.layers), self.n, B, M, Hq, Hkv, D, page_size,
                                                FP8KV_CACHE_E4M3, _ptr(self.workspace), self.workspace.numel(),
                                                _stream(stream))
        _check("fp8kv_paged_attention_layers", rc)


def fp8kv_paged_attention_layers(layers, workspace=None, stream=None):
    """Run the verifier step of several layers in one launch (see
    PagedAttentionLayers); returns the prepared call for reuse."""
    call = PagedAttentionLayers(layers, workspace)
    call(stream)
    return call


def fp8kv_e4m3_encode_bits(first: int, n: int, out: torch.Tensor, stream=None):
    _dev(out, "out", torch.uint8)
    rc = lib().fp8kv_e4m3_encode_bits(first, n, _ptr(out), _stream(stream))
    _check("fp8kv_e4m3_encode_bits", rc)


def fp8kv_selftest_bounded_wait(limit_us: int, stream=None):
    """Launch the kernel whose barrier wait runs out after limit_us (sets
    DEV_WAIT_TIMEOUT in the device status word)."""
    _check("fp8kv_selftest_bounded_wait", lib().fp8kv_selftest_bounded_wait(int(limit_us), _stream(stream)))


def fp8kv_last_dispatch() -> str:
    buf = ctypes.create_string_buffer(512)
    lib().fp8kv_last_dispatch(buf, 512)
    return buf.value.decode()


def fp8kv_launch_count():
    """Kernel launches the library has made in this process."""
    return int(lib().fp8kv_launch_count())


def fp8kv_device_status(clear: bool = False) -> int:
    s = ctypes.c_uint(0)
    _check("fp8kv_device_status", lib().fp8kv_device_status(ctypes.byref(s), int(clear)))
    return s.value
