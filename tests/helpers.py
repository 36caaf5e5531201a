"""Shared test plumbing: build the same layer on the GPU (through the C ABI) and
in the oracle (on the CPU) from one seeded input case."""
import os

import numpy as np
import torch

import oracle
from oracle import attention_np
from verify_attention_gb300 import inputs as gen

POISON_E4M3 = 0xA5          # finite (-0.203...), marks untouched slots
TOL_ABS, TOL_REL = 1e-2, 1e-2


def gpu_caches(case: gen.LayerCase, cache_dtype="e4m3", poison=POISON_E4M3, device="cuda", new_tokens=True):
    from verify_attention_gb300 import fp8kv
    lay = case.layout
    Hkv, D = case.k_new.shape[1], case.k_new.shape[2]
    shape = (lay.num_pages, Hkv, lay.page_size, D)
    if cache_dtype == "e4m3":
        kc = torch.full(shape, poison, dtype=torch.uint8, device=device)
    else:
        kc = torch.zeros(shape, dtype=torch.bfloat16, device=device)
    vc = kc.clone()
    ks = torch.tensor([case.k_scale], dtype=torch.float32, device=device)
    vs = torch.tensor([case.v_scale], dtype=torch.float32, device=device)
    parts = [(case.k_prior, case.v_prior, case.slots_prior)]
    if new_tokens:
        parts.append((case.k_new, case.v_new, case.slots_new))
    for k, v, s in parts:
        if k.shape[0]:
            fp8kv.fp8kv_cache_insert(k.to(device), v.to(device), s.to(device), ks, vs, kc, vc)
    return kc, vc, ks, vs


def _oracle_insert(k, v, slots, k_scale, v_scale, kc, vc, dt, threads):
    """oracle.cache_insert over token chunks in threads (the C call releases the
    GIL; chunks write disjoint slots)."""
    kb, vb, sb = gen.bf16_bits(k), gen.bf16_bits(v), slots.cpu().numpy()
    T = kb.shape[0]
    if threads <= 1 or T < 4096:
        oracle.cache_insert(kb, vb, sb, k_scale, v_scale, kc, vc, cache_dtype=dt)
        return
    import concurrent.futures as cf
    cuts = np.linspace(0, T, threads + 1).astype(int)
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda i: oracle.cache_insert(kb[cuts[i]:cuts[i + 1]], vb[cuts[i]:cuts[i + 1]],
                                                  sb[cuts[i]:cuts[i + 1]], k_scale, v_scale, kc, vc,
                                                  cache_dtype=dt), range(threads)))


def oracle_threads():
    return max(1, min(16, os.cpu_count() or 1))


def oracle_caches(case: gen.LayerCase, cache_dtype="e4m3", poison=POISON_E4M3, new_tokens=True):
    lay = case.layout
    Hkv, D = case.k_new.shape[1], case.k_new.shape[2]
    shape = (lay.num_pages, Hkv, lay.page_size, D)
    if cache_dtype == "e4m3":
        kc = np.full(shape, poison, np.uint8)
        dt = oracle.E4M3
    else:
        kc = np.zeros(shape, np.uint16)
        dt = oracle.BF16
    vc = kc.copy()
    parts = [(case.k_prior, case.v_prior, case.slots_prior)]
    if new_tokens:
        parts.append((case.k_new, case.v_new, case.slots_new))
    for k, v, s in parts:
        if k.shape[0]:
            _oracle_insert(k, v, s, case.k_scale, case.v_scale, kc, vc, dt, oracle_threads())
    return kc, vc


def gpu_attention(case, kc, vc, ks, vs, split_tokens=0, window_left=None, device="cuda", max_seq_len=None,
                  **kw):
    from verify_attention_gb300 import fp8kv
    lay = case.layout
    wl = case.window_left if window_left is None else window_left
    msl = int(lay.seq_lens.max()) if max_seq_len is None else max_seq_len
    return fp8kv.fp8kv_paged_attention(case.q.to(device), kc, vc, lay.block_table.to(device),
                                       lay.seq_lens.to(device), msl, ks, vs,
                                       case.sm_scale, window_left=wl, split_tokens=split_tokens, **kw)


def oracle_attention(case, kc, vc, rows=None, cache_dtype="e4m3", window_left=None, impl="c", q=None):
    """The oracle's attention for the case (every row, or the listed (b, m, h)
    rows); impl "numpy" runs the float64 numpy implementation of the same
    definition (full-size layers); q overrides the case's bf16 queries."""
    lay = case.layout
    wl = case.window_left if window_left is None else window_left
    dt = oracle.E4M3 if cache_dtype == "e4m3" else oracle.BF16
    qb = gen.bf16_bits(case.q if q is None else q)
    args = (qb, kc, vc, lay.block_table.numpy(), lay.seq_lens.numpy(), case.k_scale, case.v_scale, case.sm_scale)
    if rows is None and impl == "numpy":
        return attention_np.paged_attention(*args, window_left=wl, cache_dtype=dt)
    if rows is None:
        return oracle.paged_attention(*args, window_left=wl, cache_dtype=dt)
    return oracle.paged_attention_rows(*args, np.asarray(rows, np.int32), window_left=wl, cache_dtype=dt)


def assert_close(gpu_bf16, ref64, what=""):
    """|gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise; returns (max abs err, mean abs err)."""
    g = gpu_bf16.float().cpu().numpy().astype(np.float64) if torch.is_tensor(gpu_bf16) else gpu_bf16
    err = np.abs(g - ref64)
    bound = TOL_ABS + TOL_REL * np.abs(ref64)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()}, "
                             f"max err {np.nanmax(err):.4g}")
    return float(err.max()), float(err.mean())


def sample_rows(B, M, Hq, n, seed=0):
    rng = np.random.default_rng(seed)
    rows = set()
    # always the first and last rows of the first and last sequences
    for b in {0, B - 1}:
        for m in {0, M - 1}:
            for h in {0, Hq - 1}:
                rows.add((b, m, h))
    while len(rows) < min(n, B * M * Hq):
        rows.add((int(rng.integers(B)), int(rng.integers(M)), int(rng.integers(Hq))))
    return np.array(sorted(rows), np.int32)
