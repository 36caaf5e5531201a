"""The C-ABI library builds, loads and exports every symbol include/fp8kv.h
declares; host-side validation rejects bad arguments before any launch.
No kernel runs here (CPU only)."""
import ctypes
import os
import re

import pytest
import torch

from verify_attention_gb300 import build, fp8kv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8kv.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return fp8kv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8kv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fp8kv_cache_insert", "fp8kv_qk_norm_rope_insert", "fp8kv_paged_attention",
              "fp8kv_append_paged_attention",
              "fp8kv_paged_attention_workspace_size", "fp8kv_paged_attention_plan",
              "fp8kv_status_string", "fp8kv_last_dispatch", "fp8kv_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_selftest_limit_validation_needs_no_device(L):
    assert L.fp8kv_selftest_bounded_wait(0, NULL) == 1
    assert L.fp8kv_selftest_bounded_wait(2000001, NULL) == 1


def test_status_strings(L):
    assert fp8kv.fp8kv_status_string(0) == "ok"
    assert "unsupported" in fp8kv.fp8kv_status_string(2)
    assert "workspace" in fp8kv.fp8kv_status_string(3)
    assert fp8kv.fp8kv_status_string(99) == "unknown status"


NULL = ctypes.c_void_p(0)
P16 = ctypes.c_void_p(1 << 20)          # fake, 16-byte aligned: never dereferenced


def _attn(L, **over):
    a = dict(q=P16, k=P16, v=P16, dt=0, bt=P16, mpps=4, sl=P16, maxL=100, B=1, M=1, Hq=72, Hkv=8, D=128,
             ps=32, P=16, ks=P16, vs=P16, sm=0.088, wl=-1, split=32, ws=P16, wsb=1 << 30, out=P16,
             stream=NULL)
    a.update(over)
    return L.fp8kv_paged_attention(*a.values())


def test_attention_validation(L):
    E_INV, E_UNS, E_WS = 1, 2, 3
    assert _attn(L, q=NULL) == E_INV
    assert _attn(L, D=64) == E_UNS
    assert _attn(L, ps=16, split=0) == E_UNS
    assert _attn(L, M=17) == E_UNS
    assert _attn(L, M=0) == E_INV
    assert _attn(L, Hq=70) == E_INV                 # not a multiple of Hkv
    assert _attn(L, M=16, Hq=80) == E_UNS           # 16 x 10 rows > 144
    # more than 16 rows per sequence or 144 per KV head: E4M3 cache and whole
    # 128-key partitions only (the tcgen05 kernel's row tiles)
    assert _attn(L, M=17, dt=1, split=0) == E_UNS
    assert _attn(L, M=16, Hq=80, dt=1, split=0) == E_UNS
    assert _attn(L, M=40, split=96) == E_UNS
    assert _attn(L, M=16385, split=0) == E_UNS
    assert _attn(L, split=48) == E_INV              # not a multiple of the page size
    assert _attn(L, maxL=200) == E_INV              # beyond max_pages_per_seq * page_size
    assert _attn(L, dt=7) == E_INV
    assert _attn(L, ks=NULL) == E_INV
    assert _attn(L, q=ctypes.c_void_p((1 << 20) + 8)) == E_INV   # misaligned
    assert _attn(L, ws=NULL) == E_WS
    assert _attn(L, wsb=16) == E_WS
    assert _attn(L, wl=-2) == E_INV
    # B = 0: nothing to do, no pointer is read
    assert _attn(L, B=0, q=NULL, k=NULL, v=NULL, bt=NULL, sl=NULL, out=NULL, ws=NULL, wsb=0) == 0
    assert _attn(L, B=0, D=64) == E_UNS              # shapes are still checked


def test_append_validation(L):
    f = L.fp8kv_append_paged_attention
    a = [P16, P16, P16, P16, P16, 0, P16, 4, P16, 100, 1, 12, 72, 8, 128, 32, 16, P16, P16, 0.088, -1, 32, P16,
         1 << 30, P16, NULL]
    bad = list(a); bad[0] = NULL                   # k_new missing
    assert f(*bad) == 1
    bad = list(a); bad[1] = ctypes.c_void_p((1 << 20) + 4)   # misaligned
    assert f(*bad) == 1
    bad = list(a); bad[10] = 0; bad[0] = NULL; bad[1] = NULL   # B = 0: nothing to do
    assert f(*bad) == 0


def test_insert_validation(L):
    f = L.fp8kv_cache_insert
    args = [P16, P16, P16, 4, 8, 128, P16, P16, P16, P16, 16, 32, 0, NULL]
    bad = list(args); bad[0] = NULL
    assert f(*bad) == 1
    bad = list(args); bad[5] = 96
    assert f(*bad) == 2
    bad = list(args); bad[11] = 48
    assert f(*bad) == 2
    bad = list(args); bad[12] = 5
    assert f(*bad) == 1
    bad = list(args); bad[6] = NULL
    assert f(*bad) == 1
    bad = list(args); bad[3] = 0                    # T = 0: nothing to do
    assert f(*bad) == 0
    bad = [NULL, NULL, NULL, 0, 8, 128, NULL, NULL, NULL, NULL, 16, 32, 0, NULL]   # and no pointer is read
    assert f(*bad) == 0
    g = L.fp8kv_qk_norm_rope_insert
    a2 = [P16, P16, P16, P16, P16, P16, 1e-6, P16, 100, ctypes.c_void_p(2 << 20), P16, 4, 72, 8, 128, P16,
          P16, P16, P16, 16, 32, NULL]
    bad = list(a2); bad[9] = P16                    # q_out aliases q
    assert g(*bad) == 1
    bad = list(a2); bad[6] = -1.0
    assert g(*bad) == 1
    bad = list(a2); bad[14] = 64
    assert g(*bad) == 2


def test_per_head_entries_validation_needs_no_device(L):
    """The per-head entry points check their arguments on the host like the
    per-tensor ones (E4M3 cache implied): missing scales, sizes, B/T = 0."""
    f = L.fp8kv_cache_insert_per_head
    args = [P16, P16, P16, 4, 8, 128, P16, P16, P16, P16, 16, 32, NULL]
    assert f(*[NULL if i == 6 else a for i, a in enumerate(args)]) == 1      # k_scale missing
    assert f(*[96 if i == 5 else a for i, a in enumerate(args)]) == 2        # D != 128
    assert f(*[0 if i == 3 else a for i, a in enumerate(args)]) == 0         # T = 0
    g = L.fp8kv_paged_attention_per_head
    a = [P16, P16, P16, P16, 4, P16, 100, 1, 12, 72, 8, 128, 32, 16, P16, P16, 0.088, -1, 32, P16, 1 << 30, P16,
         NULL]
    assert g(*[NULL if i == 15 else x for i, x in enumerate(a)]) == 1        # v_scale missing
    assert g(*[64 if i == 11 else x for i, x in enumerate(a)]) == 2          # D != 128
    assert g(*[0 if i == 7 else x for i, x in enumerate(a)]) == 0            # B = 0
    h = L.fp8kv_append_paged_attention_per_head
    assert h(NULL, P16, *a) == 1                                               # k_new missing
    assert h(NULL, NULL, *[0 if i == 7 else x for i, x in enumerate(a)]) == 0


def test_per_head_binding_checks_scale_count():
    if not torch.cuda.is_available():
        k = torch.zeros(1, 8, 128, dtype=torch.bfloat16)
        with pytest.raises(ValueError):                 # CPU tensors are refused first
            fp8kv.fp8kv_cache_insert_per_head(k, k, torch.zeros(1, dtype=torch.int64), torch.ones(8), torch.ones(8),
                                              torch.zeros(1, 8, 32, 128, dtype=torch.uint8),
                                              torch.zeros(1, 8, 32, 128, dtype=torch.uint8))
        return
    k = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(1, 8, 32, 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        fp8kv.fp8kv_cache_insert_per_head(k, k, torch.zeros(1, dtype=torch.int64, device="cuda"),
                                          torch.ones(7, device="cuda"), torch.ones(8, device="cuda"), c, c)


def test_plan_and_workspace_host_logic(L):
    # explicit partitions: 131072 keys of page 64 in partitions of 2048 keys
    ns, st = fp8kv.fp8kv_paged_attention_plan(1, 1, 72, 8, 128, 64, 131072, -1, 2048)
    assert (ns, st) == (64, 2048)
    assert fp8kv.fp8kv_paged_attention_workspace_size(1, 1, 72, 8, 128, 64, 131072, -1, 2048) == \
        1 * 1 * 72 * 64 * 130 * 4
    # one partition of a decode shape: no workspace
    assert fp8kv.fp8kv_paged_attention_workspace_size(1, 1, 72, 8, 128, 64, 4096, -1, 4096) == 0
    # verifier rows in one partition: no workspace either; in two, the partials
    assert fp8kv.fp8kv_paged_attention_workspace_size(1, 12, 72, 8, 128, 64, 4096, -1, 4096) == 0
    assert fp8kv.fp8kv_paged_attention_workspace_size(1, 12, 72, 8, 128, 64, 4096, -1, 2048) == \
        1 * 12 * 72 * 2 * 130 * 4
    # a prefill chunk of 512 tokens (36 row tiles of 128 rows per KV head):
    # 288 units fill the SMs, one partition each; one KV head of a short chunk
    # gets partitions of at least 1024 keys (whole 128-key tiles)
    ns, st = fp8kv.fp8kv_paged_attention_plan(1, 512, 72, 8, 128, 64, 8192, -1, 0)
    assert (ns, st) == (1, 8192)
    ns, st = fp8kv.fp8kv_paged_attention_plan(1, 32, 9, 1, 128, 32, 32768, -1, 0)
    assert st % 128 == 0 and st >= 1024 and ns == -(-32768 // st)
    # a window of 512 with 12 rows spans at most ceil(523/64)+1 = 10 pages of 64
    ns, st = fp8kv.fp8kv_paged_attention_plan(1, 12, 72, 8, 128, 64, 8192, 511, 64)
    assert ns == 10
    with pytest.raises(fp8kv.Fp8kvError):
        fp8kv.fp8kv_paged_attention_plan(1, 1, 72, 8, 128, 64, 1000, -1, 100)


def test_automatic_plans(L):
    """The automatic partition policy on a 152-SM GB300 (the planning default
    without a device): one wave of partitions for one long sequence of
    verifier rows, one tile per partition (a cluster) when it spans at most
    8 tiles, one CTA per SM for decode, for a large batch halves of the
    longest sequence (verifier rows, taken longest first) or quarters
    (decode)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("plans depend on the device's SM count")
    plan = fp8kv.fp8kv_paged_attention_plan
    assert plan(1, 12, 72, 8, 128, 32, 8192, -1, 0) == (16, 512)     # 19 partitions max per head, whole tiles
    assert plan(1, 12, 72, 8, 128, 32, 8192, 511, 0) == (5, 128)     # window: 5 tiles -> 5-CTA cluster
    assert plan(1, 1, 72, 8, 128, 64, 131072, -1, 0) == (19, 6912)   # decode: 19 x 8 = 152 CTAs
    assert plan(64, 12, 72, 8, 128, 32, 32768, -1, 0) == (2, 16384)  # verifier batch: halves, longest first
    assert plan(64, 1, 72, 8, 128, 32, 32768, -1, 0) == (4, 8192)    # decode batch: quarters


def test_plan_invariants_over_many_shapes(L):
    """For seeded random shapes, explicit and automatic plans: whole pages per
    partition, enough partitions to cover every visible key, whole 128-key
    tiles for automatic plans (the tcgen05 kernel needs them above 16 rows per
    KV head), and a workspace exactly when a sequence spans partitions."""
    import random
    rng = random.Random(5)
    for _ in range(400):
        ps = rng.choice([32, 64])
        Hkv = rng.choice([1, 2, 8])
        G = rng.choice([1, 4, 9])
        M = rng.choice([1, 3, 12, 16, 40, 300, 1024])
        B = rng.choice([1, 3, 64])
        msl = rng.randint(M, 40000)
        wl = rng.choice([-1, 0, 63, 511])
        split = rng.choice([0, 0, ps, 4 * ps, 2048])
        ns, st = fp8kv.fp8kv_paged_attention_plan(B, M, G * Hkv, Hkv, 128, ps, msl, wl, split)
        assert ns >= 1 and st > 0 and st % ps == 0
        pages = -(-msl // ps)
        if wl >= 0:
            pages = min(pages, -(-(M + wl) // ps) + 1)
        assert ns * (st // ps) >= pages and (ns - 1) * (st // ps) < pages
        if split == 0:
            assert st % 128 == 0
        ws = fp8kv.fp8kv_paged_attention_workspace_size(B, M, G * Hkv, Hkv, 128, ps, msl, wl, split)
        assert ws == (0 if ns == 1 else B * M * G * Hkv * ns * 130 * 4)


def test_binding_rejects_cpu_tensors():
    k = torch.zeros(1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fp8kv.fp8kv_cache_insert(k, k, torch.zeros(1, dtype=torch.int64), None, None,
                                 torch.zeros(1, 8, 32, 128, dtype=torch.uint8),
                                 torch.zeros(1, 8, 32, 128, dtype=torch.uint8))


def _layer(**over):
    a = dict(q=P16, k_new=P16, v_new=P16, k_cache=P16, v_cache=P16, block_table=P16, seq_lens=P16, k_scale=P16,
             v_scale=P16, out=P16, max_pages_per_seq=4, max_seq_len=100, num_pages=16, window_left=-1,
             sm_scale=0.088)
    a.update(over)
    return fp8kv.fp8kv_layer(*a.values())


def _layers(L, layers, B=1, M=12, Hq=72, Hkv=8, D=128, ps=32, dt=0, ws=P16, wsb=1 << 30):
    arr = (fp8kv.fp8kv_layer * len(layers))(*layers)
    return L.fp8kv_paged_attention_layers(ctypes.byref(arr), len(layers), B, M, Hq, Hkv, D, ps, dt, ws, wsb, NULL)


def test_layers_entry_validation_needs_no_device(L):
    """fp8kv_paged_attention_layers rejects bad arguments before any CUDA call."""
    ok = _layer()
    assert _layers(L, [ok, _layer(q=NULL)]) == 1                     # null pointer
    assert _layers(L, [_layer(k_new=NULL)]) == 1                     # k_new without v_new
    assert _layers(L, [_layer(out=ctypes.c_void_p((1 << 20) + 8))]) == 1   # misaligned
    assert _layers(L, [_layer(max_seq_len=200)]) == 1                # beyond the block-table row
    assert _layers(L, [ok], dt=1) == 2                               # BF16 cache: not this path
    assert _layers(L, [ok], M=1) == 2                                # 9 rows per KV head: decode shape
    assert _layers(L, [ok], M=16) == 2                               # 144 rows: two row tiles
    assert _layers(L, [ok], ps=16) == 2
    assert _layers(L, [ok], wsb=100) == 3                            # workspace too small
    assert _layers(L, [ok], ws=NULL) == 3
    assert _layers(L, [ok], B=0) == 0                                # nothing to do
    assert L.fp8kv_paged_attention_layers(None, 1, 1, 12, 72, 8, 128, 32, 0, P16, 1 << 30, NULL) == 1
    need = fp8kv.fp8kv_paged_attention_layers_workspace_size(48, 1, 12, 72, 8)
    rows = 12 * 72
    assert need >= rows * 16 * (128 * 2 + 8) and need < rows * 16 * (128 * 2 + 8) + 4096
