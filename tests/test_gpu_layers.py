"""The verifier step of several layers in one persistent launch,
fp8kv_paged_attention_layers, against the oracle: the appended tokens' cache
bytes bit-exact, every output row within |err| <= 1e-2 + 1e-2 |ref| (float64
oracle), and within the same tolerance of the per-layer calls.  All calls go
through the C ABI."""
import numpy as np
import pytest
import torch

from verify_attention_gb300 import build, inputs as gen
from tests.helpers import assert_close, gpu_caches, oracle_attention, oracle_caches

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


def device_layer(case, append=True):
    """The layer's GPU tensors: the earlier context in the cache (the new tokens
    too when append is False), queries, new tokens, metadata, output."""
    kc, vc, ks, vs = gpu_caches(case, new_tokens=not append)
    lay = case.layout
    B, M = case.q.shape[0], case.M
    Hkv = case.k_new.shape[1]
    return dict(q=case.q.cuda(), k_new=case.k_new.cuda().view(B, M, Hkv, 128) if append else None,
                v_new=case.v_new.cuda().view(B, M, Hkv, 128) if append else None, k_cache=kc, v_cache=vc,
                block_table=lay.block_table.cuda(), seq_lens=lay.seq_lens.cuda(),
                max_seq_len=int(lay.seq_lens.max()), k_scale=ks, v_scale=vs, sm_scale=case.sm_scale,
                window_left=case.window_left, out=torch.full_like(case.q.cuda(), float("nan")))


def per_layer_reference(case, append=True):
    """The same layer through fp8kv_append_paged_attention (or the plain call)."""
    d = device_layer(case, append)
    f = fp8kv()
    if append:
        f.fp8kv_append_paged_attention(d["k_new"], d["v_new"], d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                       d["seq_lens"], d["max_seq_len"], d["k_scale"], d["v_scale"], d["sm_scale"],
                                       window_left=d["window_left"], out=d["out"])
    else:
        f.fp8kv_paged_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                d["max_seq_len"], d["k_scale"], d["v_scale"], d["sm_scale"],
                                window_left=d["window_left"], out=d["out"])
    return d["out"]


def check_layers(cases, appends, impl="c", compare_per_layer=True, repeat=1):
    f = fp8kv()
    layers = [device_layer(c, a) for c, a in zip(cases, appends)]
    call = f.PagedAttentionLayers(layers)
    for _ in range(repeat):
        for d in layers:
            d["out"].fill_(float("nan"))
        call()
    torch.cuda.synchronize()
    assert f.fp8kv_last_dispatch().startswith("attention_layers"), f.fp8kv_last_dispatch()
    for i, (case, d) in enumerate(zip(cases, layers)):
        okc, ovc = oracle_caches(case)
        assert np.array_equal(d["k_cache"].cpu().numpy(), okc), f"layer {i}: K cache bytes"
        assert np.array_equal(d["v_cache"].cpu().numpy(), ovc), f"layer {i}: V cache bytes"
        ref = oracle_attention(case, okc, ovc, impl=impl)
        assert_close(d["out"], ref, f"layer {i} vs oracle")
        if compare_per_layer:
            assert_close(d["out"], per_layer_reference(case, appends[i]).float().cpu().numpy().astype(np.float64),
                         f"layer {i} vs per-layer call")
    assert f.fp8kv_device_status(clear=True) == 0
    return layers


@pytest.mark.parametrize("ps", [32, 64])
def test_layers_mixed_kinds_two_sequences(ps):
    """Six layers of sliding windows of several widths and global layers, two
    sequences of different lengths (so some partitions of the shorter one are
    empty), each layer with its own pages, scales and new tokens."""
    windows = [200, None, 64, None, None, 512]
    cases = [gen.layer_case(10100 + 17 * i + ps, [900, 333], 12, ps, window=w) for i, w in enumerate(windows)]
    check_layers(cases, [True] * 6)


def test_layers_without_append_and_short_sequences():
    """Layers whose new tokens are already in the cache (no append), mixed with
    appending layers; sequences shorter than a tile and than the window."""
    cases = [gen.layer_case(10200 + i, [130, 40, 77], 12, 32, window=w)
             for i, w in enumerate([None, 512, 64, None])]
    check_layers(cases, [False, True, False, True])


@pytest.mark.parametrize("M,Hq,Hkv", [(2, 18, 2), (14, 72, 8), (4, 32, 1)])
def test_layers_row_counts(M, Hq, Hkv):
    """Row counts 18, 126 and 128 per KV head."""
    cases = [gen.layer_case(10300 + i + M, [700, 260], M, 32, window=w, Hq=Hq, Hkv=Hkv)
             for i, w in enumerate([None, 100])]
    check_layers(cases, [True, True])


def test_layers_repeated_calls_reuse_the_workspace():
    """Two calls in a row on one workspace: the counters the first call left
    at zero synchronise the second; both give the oracle's results."""
    cases = [gen.layer_case(10400 + i, [1500], 12, 64, window=w) for i, w in enumerate([None, 512, None])]
    f = fp8kv()
    layers = [device_layer(c, True) for c in cases]
    call = f.PagedAttentionLayers(layers)
    outs = []
    for _ in range(2):
        for d in layers:
            d["out"].fill_(float("nan"))
        call()
        torch.cuda.synchronize()
        outs.append([d["out"].clone() for d in layers])
    assert all(torch.equal(a, b) for a, b in zip(*outs))
    for case, d in zip(cases, layers):
        okc, ovc = oracle_caches(case)
        assert_close(d["out"], oracle_attention(case, okc, ovc), "second call")
    head = f.fp8kv_paged_attention_layers_workspace_size(3, 1, 12, 72, 8)
    assert head == call.ws_bytes
    assert int(call.workspace[:256].count_nonzero()) == 0         # counters left at zero
    assert f.fp8kv_device_status(clear=True) == 0


@pytest.mark.parametrize("ps", [32, 64])
def test_layers_verify_step_full_size(ps):
    """The 48-layer verify step ([SW512 x3, G] x12, L = 8192, M = 12) in one
    launch: every output row of every layer against the oracle (float64 numpy
    implementation), and the new tokens' cache bytes."""
    cases = [gen.cfg3_case(l, ps) for l in range(48)]
    check_layers(cases, [True] * 48, impl="numpy", compare_per_layer=False)


def test_layers_workspace_too_small_launches_nothing():
    f = fp8kv()
    case = gen.layer_case(10500, [300], 12, 32)
    d = device_layer(case, True)
    small = f.PagedAttentionLayers([d], workspace=torch.zeros(64, dtype=torch.uint8, device="cuda"))
    with pytest.raises(f.Fp8kvError) as e:
        small()
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert torch.isnan(d["out"].float()).all()                     # untouched


def test_layers_more_groups_than_sms():
    """24 sequences x 8 KV heads = 192 (sequence, KV head) groups, more than
    the 152 SMs: CTAs run several units per layer and combine after them.
    Four layers (global and sliding), ragged lengths, against the oracle and
    the per-layer calls."""
    g = torch.Generator().manual_seed(10600)
    lens = torch.randint(300, 3000, (24,), generator=g).tolist()
    cases = [gen.layer_case(10600 + i, lens, 12, 32, window=w) for i, w in enumerate([None, 512, None, 64])]
    check_layers(cases, [True] * 4, impl="numpy")


@pytest.mark.parametrize("ps", [32, 64])
def test_layers_serving_mix_shape(ps):
    """The batched serving mix's shape: 64 sequences of 1024..8192 tokens
    (2048 work units per layer over the CTAs), a global and a sliding-window
    layer: every row of every sequence against the oracle, and the cache
    bytes."""
    g = torch.Generator().manual_seed(10700 + ps)
    lens = torch.randint(1024, 8193, (64,), generator=g).tolist()
    cases = [gen.layer_case(10700 + ps + i, lens, 12, ps, window=w) for i, w in enumerate([None, 512])]
    layers = check_layers(cases, [True, True], impl="numpy", compare_per_layer=False)
    assert fp8kv().fp8kv_last_dispatch().startswith("attention_layers")
    del layers
