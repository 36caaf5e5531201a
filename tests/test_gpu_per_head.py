"""Per-head K/V scales (an extension the pages do not use: "Laguna S 2.1
KV-cache precision decision", "What the official checkpoint requests" asks for
one scale per tensor) through the C ABI against the oracle's per-head
routines: the insert bit-exact, attention within |err| <= 1e-2 + 1e-2 |ref| on
every kernel path (decode, tcgen05 with workspace reduce and with the cluster
combine, prefill row tiles, both append paths)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import attention_np
from verify_attention_gb300 import build, inputs as gen
from tests.helpers import POISON_E4M3, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    from verify_attention_gb300 import fp8kv
    fp8kv.fp8kv_device_status(clear=True)
    yield
    assert fp8kv.fp8kv_device_status(clear=True) == 0


def f():
    from verify_attention_gb300 import fp8kv
    return fp8kv


def head_case(seed, seq_lens, M, ps, window=None, Hq=72, Hkv=8):
    """A layer whose KV heads differ in magnitude by up to 8x, with the
    generator's per-head minmax scales."""
    return gen.layer_case(seed, seq_lens, M, ps, window=window, Hq=Hq, Hkv=Hkv, k_head_scale=(0.25, 2.0))


def scales(case):
    return case.k_scale_h.cuda(), case.v_scale_h.cuda()


def caches(case, new_tokens=True):
    """(GPU caches from fp8kv_cache_insert_per_head, oracle caches from
    oracle.cache_insert_per_head) over the prior (and new) tokens."""
    lay = case.layout
    Hkv = case.k_new.shape[1]
    shape = (lay.num_pages, Hkv, lay.page_size, 128)
    kc = torch.full(shape, POISON_E4M3, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    okc = np.full(shape, POISON_E4M3, np.uint8)
    ovc = okc.copy()
    ks, vs = scales(case)
    parts = [(case.k_prior, case.v_prior, case.slots_prior)]
    if new_tokens:
        parts.append((case.k_new, case.v_new, case.slots_new))
    for k, v, s in parts:
        if k.shape[0]:
            f().fp8kv_cache_insert_per_head(k.cuda(), v.cuda(), s.cuda(), ks, vs, kc, vc)
            oracle.cache_insert_per_head(gen.bf16_bits(k), gen.bf16_bits(v), s.numpy(), case.k_scale_h.numpy(),
                                         case.v_scale_h.numpy(), okc, ovc)
    return kc, vc, okc, ovc


def reference(case, okc, ovc):
    lay = case.layout
    return attention_np.paged_attention(gen.bf16_bits(case.q), okc, ovc, lay.block_table.numpy(),
                                        lay.seq_lens.numpy(), case.k_scale_h.numpy().astype(np.float64),
                                        case.v_scale_h.numpy().astype(np.float64), case.sm_scale,
                                        window_left=case.window_left)


@pytest.mark.parametrize("ps", [32, 64])
def test_per_head_insert_bit_exact(ps):
    case = head_case(7100 + ps, [300, 77], 12, ps)
    kc, vc, okc, ovc = caches(case)
    torch.cuda.synchronize()
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    # the heads really use different scales: a per-tensor insert differs
    ks1 = torch.tensor([case.k_scale], device="cuda")
    vs1 = torch.tensor([case.v_scale], device="cuda")
    kt, vt = torch.full_like(kc, POISON_E4M3), torch.full_like(vc, POISON_E4M3)
    f().fp8kv_cache_insert(case.k_prior.cuda(), case.v_prior.cuda(), case.slots_prior.cuda(), ks1, vs1, kt, vt)
    assert not torch.equal(kt, kc)


# (seq_lens, M, ps, window, split_tokens, expected kernel)
PATHS = [
    ([3000], 1, 64, None, 512, "paged_decode_mma"),       # decode, partitions + reduce
    ([900, 333], 1, 32, 200, 0, "paged_decode_mma"),      # decode, page 32, sliding
    ([1500, 700], 12, 32, None, 256, "attention_tc"),     # tcgen05, workspace reduce
    ([1000], 12, 64, None, 128, "attention_tc"),          # tcgen05, 8-CTA cluster combine
    ([640], 12, 32, 512, 0, "attention_tc"),              # tcgen05, sliding, cluster
    ([500], 40, 64, None, 0, "attention_tc"),             # prefill row tiles
]


@pytest.mark.parametrize("seq_lens,M,ps,window,split,kernel", PATHS)
def test_per_head_attention_every_path(seq_lens, M, ps, window, split, kernel):
    case = head_case(7200 + sum(seq_lens) + M, seq_lens, M, ps, window=window)
    kc, vc, okc, ovc = caches(case)
    ks, vs = scales(case)
    lay = case.layout
    out = f().fp8kv_paged_attention_per_head(case.q.cuda(), kc, vc, lay.block_table.cuda(), lay.seq_lens.cuda(),
                                             int(lay.seq_lens.max()), ks, vs, case.sm_scale,
                                             window_left=case.window_left, split_tokens=split)
    torch.cuda.synchronize()
    assert f().fp8kv_last_dispatch().startswith(kernel), f().fp8kv_last_dispatch()
    assert_close(out, reference(case, okc, ovc), "per-head attention")


@pytest.mark.parametrize("seq_lens,M,ps,window,split,kernel", [PATHS[1], PATHS[2], PATHS[3], PATHS[5]])
def test_per_head_append_every_path(seq_lens, M, ps, window, split, kernel):
    """The append variant: the new tokens' cache bytes equal the per-head
    insert's, and the output the oracle's (in-kernel append on the tcgen05
    path with one row tile, the append kernel otherwise)."""
    case = head_case(7300 + sum(seq_lens) + M, seq_lens, M, ps, window=window)
    kc, vc, _, _ = caches(case, new_tokens=False)
    _, _, okc, ovc = caches(case, new_tokens=True)
    ks, vs = scales(case)
    lay = case.layout
    B = len(seq_lens)
    Hkv = case.k_new.shape[1]
    out = f().fp8kv_append_paged_attention_per_head(
        case.k_new.cuda().view(B, M, Hkv, 128), case.v_new.cuda().view(B, M, Hkv, 128), case.q.cuda(), kc, vc,
        lay.block_table.cuda(), lay.seq_lens.cuda(), int(lay.seq_lens.max()), ks, vs, case.sm_scale,
        window_left=case.window_left, split_tokens=split)
    torch.cuda.synchronize()
    assert f().fp8kv_last_dispatch().startswith(kernel)
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    assert_close(out, reference(case, okc, ovc), "per-head append")


@pytest.mark.parametrize("M,ps,split", [(1, 64, 0), (12, 32, 0), (12, 64, 128)])
def test_equal_per_head_scales_match_the_per_tensor_call(M, ps, split):
    """Every head's scale equal to the tensor scale: bit-identical caches and
    outputs to the per-tensor entry points."""
    case = gen.layer_case(7400 + M + ps, [1200], M, ps)
    lay = case.layout
    kh = torch.full((8,), case.k_scale, dtype=torch.float32, device="cuda")
    vh = torch.full((8,), case.v_scale, dtype=torch.float32, device="cuda")
    k1, v1 = kh[:1].clone(), vh[:1].clone()
    shape = (lay.num_pages, 8, ps, 128)
    kc = torch.full(shape, POISON_E4M3, dtype=torch.uint8, device="cuda")
    vc, kc2, vc2 = kc.clone(), kc.clone(), kc.clone()
    for k, v, s in ((case.k_prior, case.v_prior, case.slots_prior), (case.k_new, case.v_new, case.slots_new)):
        f().fp8kv_cache_insert_per_head(k.cuda(), v.cuda(), s.cuda(), kh, vh, kc, vc)
        f().fp8kv_cache_insert(k.cuda(), v.cuda(), s.cuda(), k1, v1, kc2, vc2)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    args = (case.q.cuda(), kc, vc, lay.block_table.cuda(), lay.seq_lens.cuda(), int(lay.seq_lens.max()))
    a = f().fp8kv_paged_attention_per_head(*args, kh, vh, case.sm_scale, split_tokens=split)
    b = f().fp8kv_paged_attention(*args, k1, v1, case.sm_scale, split_tokens=split)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
