"""GPU parity of paged attention against the float64 oracle, within
|err| <= 1e-2 + 1e-2 |ref|.  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from verify_attention_gb300 import build, inputs as gen
from tests.helpers import assert_close, gpu_attention, gpu_caches, oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    from verify_attention_gb300 import fp8kv
    fp8kv.fp8kv_device_status(clear=True)
    yield
    assert fp8kv.fp8kv_device_status(clear=True) == 0


def fp8kv():
    from verify_attention_gb300 import fp8kv as f
    return f


def run_case(case, split_tokens=0, cache_dtype="e4m3", poison=0xA5, rows=None, impl="c"):
    kc, vc, ks, vs = gpu_caches(case, cache_dtype, poison=poison)
    out = gpu_attention(case, kc, vc, ks, vs, split_tokens=split_tokens)
    torch.cuda.synchronize()
    okc, ovc = oracle_caches(case, cache_dtype, poison=poison)
    if rows is None:
        ref = oracle_attention(case, okc, ovc, cache_dtype=cache_dtype, impl=impl)
        return out, ref, assert_close(out, ref, f"split={split_tokens}")
    ref = oracle_attention(case, okc, ovc, rows=rows, cache_dtype=cache_dtype)
    o = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    return out, ref, assert_close(o, ref, f"split={split_tokens}")


SMALL = [
    # seq_lens, M, ps, window, Hq, Hkv
    ([1, 77, 300], 1, 32, None, 72, 8),
    ([1, 77, 300], 1, 64, None, 72, 8),
    ([12, 500], 12, 64, None, 72, 8),
    ([12, 500], 12, 64, 64, 72, 8),
    ([130, 33], 12, 32, 40, 72, 8),
    ([200], 16, 32, None, 72, 8),            # 144 rows: nine row tiles
    ([95, 260], 2, 64, None, 72, 8),         # 18 rows: two row tiles, two key groups
    ([61, 300], 5, 32, 100, 72, 8),          # 45 rows: three row tiles
    ([257, 64], 3, 32, 65, 18, 2),           # the pages' per-rank shape, sliding (64, 0)
    ([257, 64], 3, 32, None, 18, 2),         # same, global (-1, -1)
    ([40], 7, 64, None, 8, 8),               # no GQA grouping
]


@pytest.mark.parametrize("seq_lens,M,ps,window,Hq,Hkv", SMALL)
@pytest.mark.parametrize("split_tokens", [0, 64, 128])
def test_attention_small_shapes(seq_lens, M, ps, window, Hq, Hkv, split_tokens):
    case = gen.layer_case(8000 + sum(seq_lens) + M, seq_lens, M, ps, window=window, Hq=Hq, Hkv=Hkv)
    run_case(case, split_tokens=split_tokens)


@pytest.mark.parametrize("M,ps", [(1, 64), (12, 32)])
def test_attention_bf16_cache(M, ps):
    case = gen.layer_case(8100 + M, [333, 70], M, ps, window=None)
    run_case(case, split_tokens=0, cache_dtype="bf16")
    run_case(case, split_tokens=ps * 2, cache_dtype="bf16")


def test_attention_stale_nan_slots_do_not_leak():
    """Unwritten slots hold the E4M3 NaN code; keys outside every row's range
    must not contribute (0 * NaN)."""
    case = gen.layer_case(8200, [45, 100], 12, 32, window=20)
    out, ref, _ = run_case(case, poison=0x7F)
    assert torch.isfinite(out.float()).all()


def test_attention_page_permutation_bit_identical():
    case = gen.layer_case(8300, [700, 129], 12, 64, window=None)
    kc, vc, ks, vs = gpu_caches(case)
    out = gpu_attention(case, kc, vc, ks, vs)
    perm = torch.randperm(kc.shape[0], generator=gen.generator(1)).cuda()
    inv = torch.argsort(perm)
    bt = case.layout.block_table
    bt2 = torch.where(bt >= 0, inv.cpu()[bt.clamp(min=0).long()].to(torch.int32), bt)
    case2 = gen.LayerCase(**{**case.__dict__, "layout": gen.PagedLayout(case.layout.page_size,
                                                                         case.layout.num_pages, bt2,
                                                                         case.layout.seq_lens)})
    out2 = gpu_attention(case2, kc[perm].contiguous(), vc[perm].contiguous(), ks, vs)
    assert torch.equal(out, out2)


def test_attention_split_agrees_with_unsplit():
    case = gen.layer_case(8400, [3000], 1, 64)
    kc, vc, ks, vs = gpu_caches(case)
    a = gpu_attention(case, kc, vc, ks, vs, split_tokens=3008 // 64 * 64 + 64).float()
    for st in (64, 256, 1024):
        b = gpu_attention(case, kc, vc, ks, vs, split_tokens=st).float()
        assert (a - b).abs().max().item() <= 1e-2


def test_attention_unvisited_pages_never_read():
    """Block-table entries of pages before every window are -1 (and so would
    read zeros if touched): the result must not change."""
    case = gen.layer_case(8500, [900], 12, 32, window=100)
    kc, vc, ks, vs = gpu_caches(case)
    out = gpu_attention(case, kc, vc, ks, vs)
    bt = case.layout.block_table.clone()
    first = (900 - 12 - 99) // 32
    bt[0, :first] = -1
    case.layout.block_table = bt
    out2 = gpu_attention(case, kc, vc, ks, vs)
    assert torch.equal(out, out2)


def test_attention_bad_seq_len_flagged():
    f = fp8kv()
    case = gen.layer_case(8600, [100], 12, 32)
    kc, vc, ks, vs = gpu_caches(case)
    case.layout.seq_lens[0] = 5                     # fewer than M = 12
    f.fp8kv_device_status(clear=True)
    gpu_attention(case, kc, vc, ks, vs, max_seq_len=100)
    assert f.fp8kv_device_status(clear=True) & f.DEV_BAD_SEQ_LEN
    case.layout.seq_lens[0] = 101                   # beyond the host's max_seq_len
    gpu_attention(case, kc, vc, ks, vs, max_seq_len=100)
    assert f.fp8kv_device_status(clear=True) & f.DEV_BAD_SEQ_LEN


def test_verifier_rows_run_on_the_tensor_memory_kernel():
    """Up to 128 rows per KV head on an E4M3 cache with partitions of whole
    128-key tiles dispatch to the tcgen05 kernel; other partitions to mma.sync."""
    case = gen.layer_case(8800, [777, 90], 12, 32, window=200)
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    ref = oracle_attention(case, okc, ovc)
    for st, kernel in ((0, "attention_tc"), (128, "attention_tc"), (256, "attention_tc"),
                       (64, "paged_attention_mma"), (96, "paged_attention_mma")):
        out = gpu_attention(case, kc, vc, ks, vs, split_tokens=st)
        assert fp8kv().fp8kv_last_dispatch().startswith(kernel), (st, fp8kv().fp8kv_last_dispatch())
        assert_close(out, ref, f"split={st}")


@pytest.mark.parametrize("L,window,split,msl,cluster", [
    (1000, None, 128, None, 8), (1000, None, 256, None, 4), (600, 200, 128, None, 2), (4096, None, 512, None, 8),
    (300, None, 128, None, 3), (500, None, 128, 1000, 8), (2000, None, 128, None, 1)])
def test_single_sequence_cluster_combine(L, window, split, msl, cluster):
    """One sequence in 2..8 partitions: the partitions of a KV head run as one
    thread-block cluster and combine in distributed shared memory (no reduce
    kernel); a larger max_seq_len leaves cluster CTAs without keys; more than
    8 partitions take the workspace partials and the reduce kernel."""
    case = gen.layer_case(9100 + L + split, [L], 12, 32, window=window)
    if msl is not None:      # room in the block table for max_seq_len (the extra entries are never read)
        bt = case.layout.block_table
        extra = -(-msl // 32) - bt.shape[1]
        case.layout.block_table = torch.cat([bt, torch.full((bt.shape[0], extra), -1, dtype=bt.dtype)], 1)
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    ref = oracle_attention(case, okc, ovc)
    out = gpu_attention(case, kc, vc, ks, vs, split_tokens=split, max_seq_len=msl)
    d = fp8kv().fp8kv_last_dispatch()
    assert d.startswith("attention_tc") and f"cluster={cluster} " in d, d
    assert ("reduce=1" in d) == (cluster == 1), d
    assert_close(out, ref, f"L={L} split={split}")


@pytest.mark.parametrize("ps,window,split", [(32, None, 128), (64, None, 256), (32, 300, 128)])
def test_longest_first_partition_order(ps, window, split):
    """Several sequences of verifier rows in several partitions: the CTAs take
    the (sequence, partition) slots longest first from an order computed on
    the device.  48 sequences of ragged lengths (some shorter than one tile,
    so most of their slots are empty; more than 512 slots at 128-key
    partitions), every row against the oracle."""
    lens = np.random.default_rng(9400 + ps).integers(12, 1500, 48).tolist()
    lens[5], lens[17] = 1500, 12
    case = gen.layer_case(9400 + ps + split, lens, 12, ps, window=window)
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    out = gpu_attention(case, kc, vc, ks, vs, split_tokens=split)
    torch.cuda.synchronize()
    d = fp8kv().fp8kv_last_dispatch()
    assert d.startswith("attention_tc") and "order=longest_first" in d and "reduce=1" in d, d
    assert_close(out, oracle_attention(case, okc, ovc), f"longest first ps={ps} split={split}")


def test_longest_first_order_flags_a_bad_length():
    """A sequence length below M in a longest-first call is flagged (by the
    order kernel) and its slots get no CTA; the other sequences are exact."""
    f = fp8kv()
    case = gen.layer_case(9450, [700, 300, 1200], 12, 32)
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    ref = oracle_attention(case, okc, ovc)
    case.layout.seq_lens[1] = 5
    f.fp8kv_device_status(clear=True)
    out = gpu_attention(case, kc, vc, ks, vs, split_tokens=256, max_seq_len=1200)
    torch.cuda.synchronize()
    assert "order=longest_first" in f.fp8kv_last_dispatch()
    assert f.fp8kv_device_status(clear=True) & f.DEV_BAD_SEQ_LEN
    assert_close(out[[0, 2]], ref[[0, 2]], "other sequences")


@pytest.mark.parametrize("M,G", [(2, 9), (2, 16), (6, 9), (8, 16), (12, 10), (16, 8), (3, 11)])
def test_tensor_memory_kernel_row_counts(M, G):
    """Row counts 18..128 through the tcgen05 kernel, both page sizes."""
    for ps in (32, 64):
        case = gen.layer_case(8900 + M + G + ps, [300, 1100], M, ps, Hq=2 * G, Hkv=2)
        kc, vc, ks, vs = gpu_caches(case)
        out = gpu_attention(case, kc, vc, ks, vs, split_tokens=256)
        assert fp8kv().fp8kv_last_dispatch().startswith("attention_tc")
        okc, ovc = oracle_caches(case)
        assert_close(out, oracle_attention(case, okc, ovc), f"M={M} G={G} ps={ps}")


def test_dispatch_marker_reports_variant():
    case = gen.layer_case(8700, [2000], 1, 64)
    kc, vc, ks, vs = gpu_caches(case)
    gpu_attention(case, kc, vc, ks, vs, split_tokens=512)
    d = fp8kv().fp8kv_last_dispatch()
    assert d.startswith("paged_decode_mma") and "ps=64" in d and "e4m3" in d and "splits=4" in d, d


@pytest.mark.parametrize("ps", [32, 64])
@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_decode_kernel_key_groups(ps, dtype):
    """M = 1 rows run on the decode kernel (several key groups, each with its
    own stages); partitions long enough for every group to take several pages,
    a ragged last page, and a partition shorter than the group count."""
    case = gen.layer_case(8750 + ps, [ps * 37 + 5, 3 * ps - 1], 1, ps)
    kc, vc, ks, vs = gpu_caches(case, cache_dtype=dtype)
    okc, ovc = oracle_caches(case, cache_dtype=dtype)
    ref = oracle_attention(case, okc, ovc, cache_dtype=dtype)
    for st in (0, ps * 16, ps * 2):
        out = gpu_attention(case, kc, vc, ks, vs, split_tokens=st)
        assert fp8kv().fp8kv_last_dispatch().startswith("paged_decode_mma")
        assert_close(out, ref, f"ps={ps} {dtype} split={st}")


@pytest.mark.parametrize("M,ps", [(1, 32), (12, 32), (12, 64)])
def test_window_of_one_key_returns_own_value(M, ps):
    """window_left = 0: every row sees only its own key, so the output is that
    key's dequantized V row (up to the bf16 output rounding), on every kernel."""
    case = gen.layer_case(9300 + M + ps, [700, 130], M, ps, window=1)
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    ref = oracle_attention(case, okc, ovc, window_left=0)
    for st in (0, ps, 4 * ps):
        out = gpu_attention(case, kc, vc, ks, vs, split_tokens=st, window_left=0)
        assert_close(out, ref, f"M={M} ps={ps} split={st}")
    # the closed form: V of position L - M + m, from the cache bytes
    lay = case.layout
    for b in range(2):
        L = int(lay.seq_lens[b])
        for m in range(M):
            pos = L - M + m
            page = int(lay.block_table[b, pos // ps])
            want = oracle.e4m3_decode(ovc[page, :, pos % ps, :]) * case.v_scale   # [Hkv][128]
            got = out[b, m].float().cpu().numpy().reshape(8, 9, 128)
            np.testing.assert_allclose(got, np.repeat(want[:, None, :], 9, 1), rtol=1e-2, atol=1e-6)


@pytest.mark.parametrize("M,G", [(2, 8), (1, 16)])
def test_sixteen_rows_fill_one_decode_tile(M, G):
    """Exactly 16 rows per KV head: the decode kernel with a full row tile."""
    case = gen.layer_case(9400 + M * G, [333, 64], M, 32, Hq=2 * G, Hkv=2)
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    out = gpu_attention(case, kc, vc, ks, vs)
    assert fp8kv().fp8kv_last_dispatch().startswith("paged_decode_mma")
    assert_close(out, oracle_attention(case, okc, ovc), f"M={M} G={G}")


def test_empty_batch_launches_nothing():
    """B = 0: the call succeeds and leaves the output untouched."""
    from verify_attention_gb300 import fp8kv as f
    q = torch.zeros(0, 12, 72, 128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros(4, 8, 32, 128, dtype=torch.uint8, device="cuda")
    bt = torch.zeros(0, 4, dtype=torch.int32, device="cuda")
    sl = torch.zeros(0, dtype=torch.int32, device="cuda")
    s = torch.ones(1, device="cuda")
    out = f.fp8kv_paged_attention(q, cache, cache, bt, sl, 128, s, s, 0.088)
    torch.cuda.synchronize()
    assert out.shape == (0, 12, 72, 128)


@pytest.mark.parametrize("seq_lens,M,ps,window,split", [
    ([700], 12, 32, None, 0),            # one sequence: one wave of partitions + reduce
    ([640], 12, 32, 512, 0),             # one sequence, sliding: cluster combine
    ([1000], 12, 32, None, 128),         # 8-CTA cluster, new tokens straddling a tile edge
    ([900], 12, 32, None, 128),          # 8-CTA cluster, new tokens in the last two partitions
    ([1163], 12, 32, 512, 0),            # sliding 5-CTA cluster, new tokens in the last two partitions
    ([300, 1000, 77], 12, 64, None, 0),  # batch, tensor-memory kernel
    ([130, 33], 12, 32, 40, 64),         # mma.sync kernel with the append kernel
    ([500, 33], 1, 64, None, 0),         # decode kernel with the append kernel
])
@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_append_equals_insert_then_attention(seq_lens, M, ps, window, split, dtype):
    """fp8kv_append_paged_attention == fp8kv_cache_insert of the new rows at
    their slots followed by fp8kv_paged_attention: identical cache bytes and
    identical outputs, and within tolerance of the oracle."""
    from verify_attention_gb300 import fp8kv as f
    case = gen.layer_case(9500 + sum(seq_lens) + M + split, seq_lens, M, ps, window=window)
    lay = case.layout
    shape = (lay.num_pages, 8, ps, 128)
    if dtype == "e4m3":
        kc = torch.full(shape, 0xA5, dtype=torch.uint8, device="cuda")
    else:
        kc = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    ks = torch.tensor([case.k_scale], device="cuda")
    vs = torch.tensor([case.v_scale], device="cuda")
    if case.k_prior.shape[0]:
        f.fp8kv_cache_insert(case.k_prior.cuda(), case.v_prior.cuda(), case.slots_prior.cuda(), ks, vs, kc, vc)
    kc2, vc2 = kc.clone(), vc.clone()
    f.fp8kv_cache_insert(case.k_new.cuda(), case.v_new.cuda(), case.slots_new.cuda(), ks, vs, kc2, vc2)
    ref = gpu_attention(case, kc2, vc2, ks, vs, split_tokens=split)
    B = len(seq_lens)
    kn = case.k_new.cuda().view(B, M, 8, 128)
    vn = case.v_new.cuda().view(B, M, 8, 128)
    out = f.fp8kv_append_paged_attention(kn, vn, case.q.cuda(), kc, vc, lay.block_table.cuda(),
                                         lay.seq_lens.cuda(), int(lay.seq_lens.max()), ks, vs, case.sm_scale,
                                         window_left=case.window_left, split_tokens=split)
    torch.cuda.synchronize()
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(out, ref)
    if dtype == "e4m3":
        okc, ovc = oracle_caches(case)
        assert np.array_equal(kc.cpu().numpy(), okc)
    else:
        okc, ovc = oracle_caches(case, "bf16")
    assert_close(out, oracle_attention(case, okc, ovc, cache_dtype=dtype), f"append {seq_lens} M={M} {dtype}")


# ---------------------------------------------- prefill-shaped row counts

PREFILL = [
    # seq_lens, M, ps, window
    ([1024], 256, 32, None),          # 2304 rows per KV head: 18 row tiles
    ([600, 300], 130, 64, 127),       # 1170 rows: 10 tiles, the last of 18 rows; sliding
    ([200], 200, 32, None),           # the whole sequence is new (L = M): causal from key 0
    ([777], 64, 64, 300),             # 576 rows, a window shorter than the chunk
]


@pytest.mark.parametrize("seq_lens,M,ps,window", PREFILL)
def test_prefill_row_tiles(seq_lens, M, ps, window):
    """More than 16 query rows per sequence (a chunk of M tokens at the end of
    the context): the tcgen05 kernel in 128-row tiles, each loading the keys
    its rows see (causal within the chunk, window), automatic and explicit
    partitions."""
    case = gen.layer_case(9700 + sum(seq_lens) + M, seq_lens, M, ps, window=window)
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    ref = oracle_attention(case, okc, ovc)
    tiles = -(-M * 9 // 128)
    for st in (0, 128, 384):
        out = gpu_attention(case, kc, vc, ks, vs, split_tokens=st)
        d = fp8kv().fp8kv_last_dispatch()
        assert d.startswith("attention_tc") and f"row_tiles={tiles} " in d, d
        assert_close(out, ref, f"prefill {seq_lens} M={M} split={st}")


def test_prefill_rows_need_e4m3_cache_and_whole_tiles():
    """Prefill row counts run only on the tcgen05 kernel: a BF16 cache or
    partitions that are not whole 128-key tiles are refused, not served slowly."""
    f = fp8kv()
    case = gen.layer_case(9750, [300], 40, 32)
    kc, vc, ks, vs = gpu_caches(case, "bf16")
    with pytest.raises(f.Fp8kvError):
        gpu_attention(case, kc, vc, ks, vs)
    kc, vc, ks, vs = gpu_caches(case)
    with pytest.raises(f.Fp8kvError):
        gpu_attention(case, kc, vc, ks, vs, split_tokens=96)


def test_prefill_append_equals_insert_then_attention():
    """A prefill chunk through the append entry (the append kernel, then the
    row-tiled attention): cache bytes of the insert, bit-identical output,
    within tolerance of the oracle."""
    from verify_attention_gb300 import fp8kv as f
    seq_lens, M, ps = [900, 400], 300, 32
    case = gen.layer_case(9760, seq_lens, M, ps)
    lay = case.layout
    kc = torch.full((lay.num_pages, 8, ps, 128), 0xA5, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    ks = torch.tensor([case.k_scale], device="cuda")
    vs = torch.tensor([case.v_scale], device="cuda")
    f.fp8kv_cache_insert(case.k_prior.cuda(), case.v_prior.cuda(), case.slots_prior.cuda(), ks, vs, kc, vc)
    kc2, vc2 = kc.clone(), vc.clone()
    f.fp8kv_cache_insert(case.k_new.cuda(), case.v_new.cuda(), case.slots_new.cuda(), ks, vs, kc2, vc2)
    ref = gpu_attention(case, kc2, vc2, ks, vs)
    B = len(seq_lens)
    out = f.fp8kv_append_paged_attention(case.k_new.cuda().view(B, M, 8, 128), case.v_new.cuda().view(B, M, 8, 128),
                                         case.q.cuda(), kc, vc, lay.block_table.cuda(), lay.seq_lens.cuda(),
                                         int(lay.seq_lens.max()), ks, vs, case.sm_scale)
    torch.cuda.synchronize()
    assert "row_tiles=22 " in f.fp8kv_last_dispatch()
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(out, ref)
    okc, ovc = oracle_caches(case)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert_close(out, oracle_attention(case, okc, ovc), "prefill append")


@pytest.mark.parametrize("M,window", [(12, None), (12, 512), (1, None)])
def test_unit_scale_draft_cache_layer(M, window):
    """The draft model's cache layers hold E4M3 with K/V scales of exactly 1.0
    (no calibration): the codes are the bf16 values rounded onto the E4M3
    grid as they are (bit-exact against the oracle), and attention over them
    stays within tolerance."""
    case = gen.layer_case(9800 + M + (window or 0), [700, 260], M, 32, window=window)
    case = gen.LayerCase(**{**case.__dict__, "k_scale": 1.0, "v_scale": 1.0})
    kc, vc, ks, vs = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    out = gpu_attention(case, kc, vc, ks, vs)
    assert_close(out, oracle_attention(case, okc, ovc), f"unit scale M={M} window={window}")


# ------------------------------------------------------------ the configs
#
# The five workloads at their full sizes.  Where the bench runs a layer
# through the one-call append entry (new tokens into the cache, then
# attention, automatic partitions), so does the test; every output row is
# compared with the oracle (the float64 numpy implementation where the C loops
# would take minutes), except on the serving mix, which is checked on every row
# of 8 whole sequences and of one KV head of each other sequence per layer.


def run_append_case(case, split_tokens=0, cache_dtype="e4m3", impl="numpy"):
    """Context inserted, then fp8kv_append_paged_attention of the new tokens:
    cache bytes bit-exact against the oracle's insert of every token, every
    output row within tolerance of the oracle."""
    f = fp8kv()
    kc, vc, ks, vs = gpu_caches(case, cache_dtype, new_tokens=False)
    lay = case.layout
    B, M = case.q.shape[0], case.M
    Hkv = case.k_new.shape[1]
    out = f.fp8kv_append_paged_attention(case.k_new.cuda().view(B, M, Hkv, 128), case.v_new.cuda().view(B, M, Hkv, 128),
                                         case.q.cuda(), kc, vc, lay.block_table.cuda(), lay.seq_lens.cuda(),
                                         int(lay.seq_lens.max()), ks, vs, case.sm_scale,
                                         window_left=case.window_left, split_tokens=split_tokens)
    torch.cuda.synchronize()
    okc, ovc = oracle_caches(case, cache_dtype)
    if cache_dtype == "bf16":
        gk, gv = gen.bf16_bits(kc), gen.bf16_bits(vc)
    else:
        gk, gv = kc.cpu().numpy(), vc.cpu().numpy()
    assert np.array_equal(gk, okc) and np.array_equal(gv, ovc)
    ref = oracle_attention(case, okc, ovc, cache_dtype=cache_dtype, impl=impl)
    return out, ref, assert_close(out, ref, f"append split={split_tokens}")


def test_cfg1_tiny_decode():
    run_case(gen.cfg1_case())
    run_append_case(gen.cfg1_case(), impl="c")


@pytest.mark.parametrize("window", [None, 512])
def test_cfg2_single_layer_verify(window):
    run_case(gen.cfg2_case(window))
    run_append_case(gen.cfg2_case(window))


@pytest.mark.parametrize("ps", [32, 64])
@pytest.mark.parametrize("layer", [0, 3])        # sliding, global
def test_cfg3_verify_layers(layer, ps):
    """A sliding and a global layer of the 48-layer step at both page sizes:
    every one of the 864 output rows, through the append entry the bench
    times (automatic partitions: a 5-CTA cluster on the sliding layer, 16
    partitions and the reduce kernel on the global one)."""
    run_append_case(gen.cfg3_case(layer, ps))


@pytest.mark.parametrize("split_tokens", [2048, 0])
def test_cfg4_long_context_decode_full_size(split_tokens):
    case = gen.cfg4_case(0)
    run_case(case, split_tokens=split_tokens, impl="numpy")
    if split_tokens == 0:
        run_append_case(case)


def test_cfg4_bf16_cache_full_size():
    run_case(gen.cfg4_case(1), split_tokens=2048, cache_dtype="bf16", impl="numpy")
    run_append_case(gen.cfg4_case(1), cache_dtype="bf16")


def cfg5_subset(layer, lens, full_count=8, Hkv=8):
    """The serving mix's checked rows on one layer: every KV head of 8 seeded
    whole sequences (the shortest and the longest always among them), and one
    seeded KV head of every other sequence."""
    rng = np.random.default_rng(5000 + layer)
    order = np.argsort(lens)
    full = {int(order[0]), int(order[-1])}
    for b in rng.permutation(len(lens)):
        if len(full) == full_count:
            break
        full.add(int(b))
    groups = [(b, hk) for b in sorted(full) for hk in range(Hkv)]
    groups += [(b, int(rng.integers(Hkv))) for b in range(len(lens)) if b not in full]
    return groups


@pytest.mark.parametrize("layer", range(8))      # G, SW, G, SW, ...
def test_cfg5_serving_mix_full_size(layer):
    """Config 5 as the bench runs it, on every layer: 64 sequences of 1024 to
    32768 tokens in one shared page-32 pool, the 12 new tokens of each through
    the fused Q/K RMSNorm + RoPE + E4M3 insert, then attention over the normed,
    rotated queries (automatic partitions).  Q and the whole cache bit-exact;
    attention on the rows of cfg5_subset."""
    import oracle
    from oracle import attention_np
    f = fp8kv()
    lens = gen.cfg5_seq_lens()
    case = gen.cfg5_case(layer, device="cuda", seq_lens=lens)
    fc = gen.fused_case(1005 * 100 + 50 + layer, case.layout, 12)
    lay = case.layout
    kc, vc, ks, vs = gpu_caches(case, new_tokens=False)
    q_out = torch.empty(fc.q.shape, dtype=torch.bfloat16, device="cuda")
    f.fp8kv_qk_norm_rope_insert(fc.q.cuda(), fc.k.cuda(), fc.v.cuda(), fc.positions.cuda(), fc.q_norm_w.cuda(),
                                fc.k_norm_w.cuda(), fc.eps, fc.cos_sin.cuda(), q_out, fc.slots.cuda(), ks, vs, kc, vc)
    q = q_out.view(len(lens), 12, 72, 128)
    out = f.fp8kv_paged_attention(q, kc, vc, lay.block_table.cuda(), lay.seq_lens.cuda(), max(lens), ks, vs,
                                  case.sm_scale, window_left=case.window_left)
    torch.cuda.synchronize()
    okc, ovc = oracle_caches(case, new_tokens=False)
    oq = oracle.qk_norm_rope_insert(gen.bf16_bits(fc.q), gen.bf16_bits(fc.k), gen.bf16_bits(fc.v),
                                    fc.positions.numpy(), gen.bf16_bits(fc.q_norm_w), gen.bf16_bits(fc.k_norm_w),
                                    fc.eps, fc.cos_sin.numpy(), fc.slots.numpy(), case.k_scale, case.v_scale,
                                    okc, ovc)
    assert np.array_equal(gen.bf16_bits(q_out), oq)
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    groups = cfg5_subset(layer, lens)
    ref = attention_np.paged_attention_groups(oq.reshape(len(lens), 12, 72, 128), okc, ovc,
                                              lay.block_table.numpy(), lay.seq_lens.numpy(), case.k_scale,
                                              case.v_scale, case.sm_scale, groups, window_left=case.window_left)
    o = out.float().cpu().numpy()
    for (b, hk), r in ref.items():
        assert_close(o[b, :, hk * 9:(hk + 1) * 9, :], r, f"layer {layer} sequence {b} (L={lens[b]}) KV head {hk}")
    assert len(ref) == 8 * 8 + 56
