"""Algorithmic bytes and flops of the hot path (what the method must move).

The per-token payload is the one printed on "Laguna S 2.1 KV-cache precision
decision", section "BF16 versus FP8 in concrete terms": K + V = 2 x 8 heads x
128 values per token per layer, 1 byte each in E4M3, 2 in BF16.  Split-KV
scratch, padding rows and re-reads are implementation overhead and are not
counted.
"""
from __future__ import annotations

from typing import Iterable


def kv_bytes_per_token_layer(Hkv: int = 8, D: int = 128, elem_bytes: int = 1) -> int:
    return 2 * Hkv * D * elem_bytes


def visible_keys_any_row(L: int, M: int, window_left: int) -> int:
    """Distinct keys visible to at least one of the M rows of a sequence of
    length L (rows at positions L-M .. L-1)."""
    if window_left < 0:
        return L
    return min(L, window_left + M)


def visible_keys_row(L: int, M: int, m: int, window_left: int) -> int:
    p = L - M + m
    lo = 0 if window_left < 0 else max(0, p - window_left)
    return p - lo + 1


def attention_bytes(seq_lens: Iterable[int], M: int, Hq: int, Hkv: int, D: int,
                    elem_bytes: int, window_left: int, page_size: int) -> int:
    """KV pages read once + Q read + O written (bf16) + block-table/seq_len/scale
    metadata (4 B per page touched, 4 B per sequence, 8 B of scales)."""
    total = 8
    for L in seq_lens:
        U = visible_keys_any_row(L, M, window_left)
        pages = -(-U // page_size) + 1
        total += U * Hkv * D * 2 * elem_bytes + 2 * M * Hq * D * 2 + 4 * pages + 4
    return total


def attention_flops(seq_lens: Iterable[int], M: int, Hq: int, D: int, window_left: int) -> int:
    """Useful flops: 2*D for Q.K and 2*D for P.V per (row, head, visible key)."""
    f = 0
    for L in seq_lens:
        for m in range(M):
            f += 4 * D * Hq * visible_keys_row(L, M, m, window_left)
    return f


def insert_bytes(T: int, Hkv: int, D: int, elem_bytes: int = 1) -> int:
    """Read bf16 K and V, write the cache elements, read the int64 slot."""
    return T * Hkv * D * 2 * (2 + elem_bytes) + 8 * T


def fused_insert_bytes(T: int, Hq: int, Hkv: int, D: int) -> int:
    """Insert plus Q read and written in bf16, the int64 position, one fp32
    cos/sin row per token and both bf16 norm weights."""
    return insert_bytes(T, Hkv, D, 1) + T * Hq * D * 2 * 2 + 8 * T + T * D * 4 + 2 * D * 2
