"""The allocation-free attention entry point, fp8kv_paged_attention_noalloc.

Some callers cannot allocate device memory at the moment they run attention:
a serving loop that must not call an allocator between steps, a process whose
memory pool is already fully carved up, or host code that holds only a raw
stream and no allocator.  For them the library keeps the split-KV partials in
a fixed device buffer of its own (32 MiB, held by every GPU that loads the
library) instead of a caller-provided workspace.

These tests call that entry point through the C ABI and compare it with the
entry point that takes a caller-provided workspace, within the tolerance the
parity tests use, on two calls in a row with different shapes (the shared
buffer keeps the previous call's contents, which must not leak into the next
result).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from verify_attention_gb300 import build, inputs as gen
from tests.helpers import TOL_ABS, TOL_REL, gpu_caches, gpu_attention


def _lib():
    build.build()
    from verify_attention_gb300 import fp8kv
    return fp8kv


def _noalloc(f, case, kc, vc, ks, vs, split_tokens):
    lay = case.layout
    out = torch.full(case.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    f.fp8kv_paged_attention_noalloc(case.q.cuda(), kc, vc, lay.block_table.cuda(), lay.seq_lens.cuda(),
                                    int(lay.seq_lens.max()), ks, vs, case.sm_scale, out,
                                    window_left=case.window_left, split_tokens=split_tokens)
    return out


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(a - b) <= TOL_ABS + TOL_REL * np.abs(b))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    f = _lib()
    f.fp8kv_device_status(clear=True)
    cases = [(gen.layer_case(9101, [5000], 1, 64), 256),               # decode, 20 partitions
             (gen.layer_case(9102, [900, 333], 12, 32, window=300), 64)]  # verifier, sliding window
    built = [(c, st, *gpu_caches(c)) for c, st in cases]
    for case, st, kc, vc, ks, vs in built:
        ref = gpu_attention(case, kc, vc, ks, vs, split_tokens=st)
        got = _noalloc(f, case, kc, vc, ks, vs, st)
        _close(got, ref)
        assert "splits=1 " not in f.fp8kv_last_dispatch()           # the shared buffer was used
    # and the first shape again, after the second one overwrote the buffer
    case, st, kc, vc, ks, vs = built[0]
    _close(_noalloc(f, case, kc, vc, ks, vs, st), gpu_attention(case, kc, vc, ks, vs, split_tokens=st))
    assert f.fp8kv_device_status(clear=True) == 0


@pytest.mark.gpu
def test_noalloc_single_sequence_cluster_path():
    """One sequence of verifier rows in at most 8 partitions: the partitions of
    a KV head combine on chip as a thread-block cluster.  The call still gets
    the shared buffer's address (the workspace is reserved for that shape), so
    it runs through the allocation-free entry point too, twice in a row."""
    f = _lib()
    f.fp8kv_device_status(clear=True)
    case = gen.layer_case(9103, [1000], 12, 32)                   # 8 tiles of 128 keys
    kc, vc, ks, vs = gpu_caches(case)
    ref = gpu_attention(case, kc, vc, ks, vs)
    assert "cluster=8 " in f.fp8kv_last_dispatch()
    for _ in range(2):
        got = _noalloc(f, case, kc, vc, ks, vs, 0)
        assert "cluster=8 " in f.fp8kv_last_dispatch()
        _close(got, ref)
    assert f.fp8kv_device_status(clear=True) == 0


@pytest.mark.gpu
def test_noalloc_rejects_requests_beyond_its_buffer():
    f = _lib()
    L = f.lib()
    # 64 sequences x 12 rows x 72 heads with 256-key partitions of 32k keys needs far more than 32 MiB
    need = f.fp8kv_paged_attention_workspace_size(64, 12, 72, 8, 128, 32, 32768, -1, 256)
    assert need > (32 << 20)
    p = ctypes.c_void_p(1 << 20)
    rc = L.fp8kv_paged_attention_noalloc(p, p, p, 0, p, 1024, p, 32768, 64, 12, 72, 8, 128, 32, 70000, p, p,
                                         0.088, -1, 256, p, None)
    assert rc == 3   # FP8KV_ERR_WORKSPACE, nothing launched
    # an invalid request that is also too large reports the invalid argument
    rc = L.fp8kv_paged_attention_noalloc(None, p, p, 0, p, 1024, p, 32768, 64, 12, 72, 8, 128, 32, 70000, p, p,
                                         0.088, -1, 256, p, None)
    assert rc == 1   # FP8KV_ERR_INVALID_ARG
    # the binding refuses an output buffer smaller than q
    case = gen.layer_case(9104, [300], 12, 32)
    kc, vc, ks, vs = gpu_caches(case)
    lay = case.layout
    with pytest.raises(ValueError):
        f.fp8kv_paged_attention_noalloc(case.q.cuda(), kc, vc, lay.block_table.cuda(), lay.seq_lens.cuda(), 300,
                                        ks, vs, case.sm_scale, torch.empty(1, 12, 72, 64, dtype=torch.bfloat16,
                                                                           device="cuda"))
