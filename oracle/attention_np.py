"""float64 paged attention in numpy -- TEST INFRASTRUCTURE.

The same definition as ``oracle_paged_attention`` in ``fp8kv_oracle.c``, for
the parity checks at full workload sizes, where the C oracle's one-element-
at-a-time loops would take hours:

    Kd = decode(k_code) * k_scale,  Vd = decode(v_code) * v_scale
    (k_scale, v_scale: scalars, or per-head arrays [Hkv] -- an extension the
    pages do not use -- whose entry hk scales KV head hk)
    out[b][m][h] = softmax_j( (q . Kd_j) * sm_scale ) . Vd      over visible j

"Exact q1/M12 paged attention" over the E4M3 cache ("Laguna S 2.1 INT4 --
calibrated FP8 KV on Intel B70", section "Initial optimization order", item 2)
with "scale/dequantize" on read ("Laguna S 2.1 KV-cache precision decision",
property table, row "Cache write/read work").  Row m of sequence b sits at
position p = L - M + m and sees keys lo..p, lo = max(0, p - window_left) for a
sliding layer, 0 for a global one; query head h reads KV head h // (Hq/Hkv).

Steps, per (sequence, KV head): gather the codes of the keys any of its rows
sees through the block table and decode them with the C oracle's E4M3 decoder
(its 256 values); then per query row, over that row's visible keys only: one
matrix product for the logits of the row's G heads, the textbook
max-subtracted softmax, one matrix product with the values.  numpy's
matrix product is the only library step.  Only ``tests/``, the smoke check and
the bench's CPU baseline leg may use this module; the product never does.
"""
from __future__ import annotations

import numpy as np

E4M3, BF16 = 0, 1


def _decode_table():
    from . import e4m3_decode
    return e4m3_decode(np.arange(256, dtype=np.uint8))


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _scale_of(scale, hk):
    """A scalar scale, or head hk's entry of per-head scales [Hkv]."""
    a = np.asarray(scale, np.float64).reshape(-1)
    return float(a[0] if a.shape[0] == 1 else a[hk])


def _rows_of_group(q_bits, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, sm_scale, b, hk,
                   window_left, cache_dtype, table):
    """float64 [M][G][D]: every query row of KV head hk of sequence b."""
    _, M, Hq, D = q_bits.shape
    num_pages, Hkv, ps, _ = k_cache.shape
    G = Hq // Hkv
    L = int(seq_lens[b])
    if L < M or -(-L // ps) > block_table.shape[1]:
        raise ValueError("sequence length outside the block table")
    out = np.empty((M, G, D), np.float64)
    qg = _bf16_to_f64(q_bits[b, :, hk * G:(hk + 1) * G, :])             # [M][G][D]
    pos = [L - M + m for m in range(M)]
    lo = [max(0, p - window_left) if window_left >= 0 else 0 for p in pos]
    # the keys any row of the group sees, dequantized once
    j0, j1 = min(lo), max(pos)
    keys = np.arange(j0, j1 + 1)
    pages = block_table[b, keys // ps]
    offs = keys % ps
    pg = np.clip(pages, 0, num_pages - 1)        # a row whose keys touch a bad page is refused below
    if cache_dtype == E4M3:
        kd = table[k_cache[pg, hk, offs, :]] * _scale_of(k_scale, hk)   # [n][D]
        vd = table[v_cache[pg, hk, offs, :]] * _scale_of(v_scale, hk)
    else:
        kd = _bf16_to_f64(k_cache[pg, hk, offs, :])
        vd = _bf16_to_f64(v_cache[pg, hk, offs, :])
    for m in range(M):
        vis = slice(lo[m] - j0, pos[m] - j0 + 1)                         # keys lo .. p of this row
        if (pages[vis] < 0).any() or (pages[vis] >= num_pages).any():
            raise ValueError("a visible key's page is outside the cache")
        s = (qg[m] @ kd[vis].T) * float(sm_scale)                        # [G][n]
        w = np.exp(s - s.max(axis=1, keepdims=True))
        out[m] = (w @ vd[vis]) / w.sum(axis=1, keepdims=True)
    return out


def paged_attention_groups(q_bits, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, sm_scale, groups,
                           window_left=-1, cache_dtype=E4M3):
    """{(b, hk): float64 [M][G][D]} for the listed (sequence, KV head) groups."""
    q_bits = np.asarray(q_bits, np.uint16)
    block_table = np.asarray(block_table, np.int64)
    seq_lens = np.asarray(seq_lens, np.int64)
    table = _decode_table() if cache_dtype == E4M3 else None
    return {(int(b), int(hk)): _rows_of_group(q_bits, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale,
                                              sm_scale, int(b), int(hk), int(window_left), cache_dtype, table)
            for b, hk in groups}


def paged_attention(q_bits, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, sm_scale, window_left=-1,
                    cache_dtype=E4M3):
    """float64 [B][M][Hq][D], every row (the C oracle's paged_attention)."""
    B, M, Hq, D = np.asarray(q_bits).shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    res = paged_attention_groups(q_bits, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale, sm_scale,
                                 [(b, hk) for b in range(B) for hk in range(Hkv)], window_left, cache_dtype)
    out = np.empty((B, M, Hq, D), np.float64)
    for (b, hk), o in res.items():
        out[b, :, hk * G:(hk + 1) * G, :] = o
    return out
