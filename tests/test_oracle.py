"""Pins of the CPU oracle against things other than itself: the E4M3 format
table, a brute-force grid search, torch's float8_e4m3fn cast, hand-worked
fixtures, closed forms, invariants and torch's float64 SDPA.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_np
from verify_attention_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(x):
    return np.float32(x)


def bits_to_f32(u):
    return np.array(u, dtype=np.uint32).view(np.float32)


# ----------------------------------------------------------------- decode

def test_decode_matches_format_table():
    for line in open(os.path.join(GOLDEN, "e4m3fn_codes.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()
        got = oracle.e4m3_decode(np.array([int(code, 16)], np.uint8))[0]
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_decode_all_codes_match_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert nan.sum() == 2  # only S.1111.111


def test_decode_grid_structure():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448
    assert np.all(np.diff(v) > 0)
    # subnormal spacing 2^-9 for the first 8 codes, then 8 steps per binade
    assert np.allclose(np.diff(v[:9]), 2.0 ** -9)
    for e in range(1, 16):
        lo = 8 * e
        step = np.diff(v[lo:min(lo + 9, 0x7F)])
        assert np.allclose(step, 2.0 ** (e - 7 - 3))
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -v)


# ----------------------------------------------------------------- encode

def test_encode_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_midpoints_ties_to_even():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        mid = f32((v[c] + v[c + 1]) / 2)           # exact in fp32
        assert float(mid) == (v[c] + v[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(np.array([mid]))[0] == even
        assert oracle.e4m3_encode(np.array([-mid]))[0] == even | 0x80
        below = np.nextafter(mid, f32(0))
        above = np.nextafter(mid, f32(1e9))
        assert oracle.e4m3_encode(np.array([below]))[0] == c
        assert oracle.e4m3_encode(np.array([above]))[0] == c + 1


def test_encode_saturation_nan_zero():
    big = np.array([448.0, np.nextafter(f32(448), f32(1e9)), 463.9, 464.0, 500.0, 1e30,
                    np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    nan = bits_to_f32([0x7FC00000, 0xFFC00000, 0x7F800001])
    assert list(oracle.e4m3_encode(nan)) == [0x7F, 0xFF, 0x7F]
    z = np.array([0.0, -0.0, 1e-40, -1e-40, 2.0 ** -11, -(2.0 ** -11)], np.float32)
    assert list(oracle.e4m3_encode(z)) == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]
    # just above half the smallest subnormal rounds up to it
    assert oracle.e4m3_encode(np.array([np.nextafter(f32(2.0 ** -10), f32(1))]))[0] == 0x01
    assert oracle.e4m3_encode(np.array([f32(2.0 ** -10)]))[0] == 0x00  # tie -> even (0)


def _brute_force_encode(x):
    """Nearest point of the 127 non-negative finite E4M3 values, ties to the even
    code, saturating; independent of the oracle's integer rounding."""
    grid = np.array([(1 + (c & 7) / 8) * 2.0 ** ((c >> 3) - 7) if (c >> 3) else (c & 7) * 2.0 ** -9
                     for c in range(0x7F)])
    a = np.abs(x.astype(np.float64))
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    idx = np.where(cand.sum(1) > 1, np.argmax(cand & (np.arange(0x7F) % 2 == 0), 1), np.argmin(d, 1))
    idx = np.where(a >= 448.0, 0x7E, idx)
    return (idx | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def test_encode_vs_brute_force_grid_search():
    rng = np.random.default_rng(5)
    mag = 2.0 ** rng.uniform(-13, 9.5, 20000)
    x = (mag * rng.choice([-1, 1], 20000)).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _brute_force_encode(x))


def test_encode_bits_range_matches_array_encoder():
    first = 0x3F7F0000
    x = (np.arange(1 << 16, dtype=np.uint32) + np.uint32(first)).view(np.float32)
    assert np.array_equal(oracle.e4m3_encode_bits(first, 1 << 16), oracle.e4m3_encode(x))


def test_encode_vs_torch_cast_in_range():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(100000) * 50).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


# ----------------------------------------------------------------- insert

def test_insert_hand_case():
    D, Hkv, ps, P = 128, 2, 4, 3
    k = np.zeros((3, Hkv, D), np.float32)
    v = np.zeros((3, Hkv, D), np.float32)
    k[0, 0, 0], k[0, 1, 5] = 0.5, -3.0       # with k_scale 0.25: 2.0, -12.0
    k[1, 0, 127] = 1000.0                      # saturates
    v[0, 1, 7] = 0.75                          # with v_scale 0.5: 1.5
    kb = torch.from_numpy(k).to(torch.bfloat16)
    vb = torch.from_numpy(v).to(torch.bfloat16)
    kc = np.full((P, Hkv, ps, D), 0xA5, np.uint8)
    vc = np.full((P, Hkv, ps, D), 0xA5, np.uint8)
    slots = np.array([9, 2, -1], np.int64)     # token 2 skipped
    oracle.cache_insert(gen.bf16_bits(kb), gen.bf16_bits(vb), slots, 0.25, 0.5, kc, vc)
    assert kc[2, 0, 1, 0] == 0x40 and kc[2, 1, 1, 5] == 0xD4   # 2.0 ; -12.0 = 1.1010.100
    assert kc[0, 0, 2, 127] == 0x7E
    assert vc[2, 1, 1, 7] == 0x3C                              # 1.5 = 0 0111 100
    assert kc[2, 0, 1, 1] == 0x00 and vc[0, 0, 2, 0] == 0x00
    touched = np.zeros_like(kc, bool)
    touched[2, :, 1, :] = True
    touched[0, :, 2, :] = True
    assert np.all(kc[~touched] == 0xA5) and np.all(vc[~touched] == 0xA5)


def test_insert_bf16_cache_copies_bits():
    g = gen.generator(3)
    k = gen.bf16_normal((5, 2, 128), g)
    v = gen.bf16_normal((5, 2, 128), g)
    kc = np.zeros((4, 2, 8, 128), np.uint16)
    vc = np.zeros((4, 2, 8, 128), np.uint16)
    slots = np.array([0, 31, 8, -5, 17], np.int64)
    oracle.cache_insert(gen.bf16_bits(k), gen.bf16_bits(v), slots, 1.0, 1.0, kc, vc,
                        cache_dtype=oracle.BF16)
    kb = gen.bf16_bits(k)
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(kc[s // 8, :, s % 8, :], kb[t])


# ------------------------------------------------------------ RMSNorm/RoPE

def test_rope_table_against_generator_and_closed_values():
    ours = oracle.rope_table(1e6, 300, 128)
    theirs = gen.rope_cos_sin(1e6, 300, 128).numpy()
    ulps = np.abs(ours.view(np.int32).astype(np.int64) - theirs.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1
    assert np.all(ours[0, :64] == 1.0) and np.all(ours[0, 64:] == 0.0)
    assert ours[1, 0] == f32(math.cos(1.0)) and ours[1, 64] == f32(math.sin(1.0))
    # the slowest frequency is theta^(-126/128)
    assert abs(ours[299, 127] - math.sin(299 * 1e6 ** (-126 / 128))) < 1e-7
    assert np.allclose(ours[:, :64] ** 2 + ours[:, 64:] ** 2, 1.0, atol=1e-6)


def test_norm_rope_worked_fixture():
    x = np.zeros(128, np.uint16)
    x[0] = 0x3F80                               # bf16 1.0
    w = np.full(128, 0x3F80, np.uint16)
    table = oracle.rope_table(1e6, 2, 128)
    want = {}
    for line in open(os.path.join(GOLDEN, "rope_worked.txt")):
        if line.strip() and not line.startswith("#"):
            p, d, val = line.split()
            want[(int(p), int(d))] = float(val)
    for pos in (0, 1):
        out = oracle.norm_rope_row(x, w, 1e-6, table[pos])
        outf = (out.astype(np.uint32) << 16).view(np.float32)
        for d in range(128):
            assert outf[d] == want.get((pos, d), 0.0), (pos, d)


def _norm_ref64(x, w, eps=1e-6):
    x = x.astype(np.float64)
    return x / np.sqrt(np.mean(x * x) + eps) * w


def test_norm_rope_against_float64_definition():
    g = gen.generator(11)
    x = gen.bf16_normal((40, 128), g)
    w = (0.5 + torch.rand((128,), generator=g)).to(torch.bfloat16)
    table = oracle.rope_table(1e6, 4096, 128)
    xs, ws = gen.bf16_bits(x), gen.bf16_bits(w)
    xf, wf = x.float().numpy(), w.float().numpy()
    for i in range(40):
        pos = 97 * i
        out = oracle.norm_rope_row(xs[i], ws, 1e-6, table[pos])
        outf = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        y = _norm_ref64(xf[i], wf)
        c, s = table[pos, :64].astype(np.float64), table[pos, 64:].astype(np.float64)
        ref = np.concatenate([y[:64] * c - y[64:] * s, y[64:] * c + y[:64] * s])
        assert np.allclose(outf, ref, rtol=2 ** -6, atol=2 ** -6)


def test_norm_rope_constant_vector_and_relative_position():
    w1 = np.full(128, 0x3F80, np.uint16)
    table = oracle.rope_table(1e6, 64, 128)
    for val in (0x3F80, 0xC000, 0x3E00):       # 1.0, -2.0, 0.125
        x = np.full(128, val, np.uint16)
        out = oracle.norm_rope_row(x, w1, 1e-6, table[0])
        outf = (out.astype(np.uint32) << 16).view(np.float32)
        assert np.all(np.abs(outf) == 1.0)
    g = gen.generator(12)
    q = gen.bf16_bits(gen.bf16_normal((128,), g))
    k = gen.bf16_bits(gen.bf16_normal((128,), g))

    def dot(a, b):
        fa = (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        fb = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return float(fa @ fb)
    d0 = dot(oracle.norm_rope_row(q, w1, 1e-6, table[10]), oracle.norm_rope_row(k, w1, 1e-6, table[3]))
    d1 = dot(oracle.norm_rope_row(q, w1, 1e-6, table[40]), oracle.norm_rope_row(k, w1, 1e-6, table[33]))
    assert abs(d0 - d1) < 0.02 * 128 ** 0.5


def test_fused_insert_equals_composition():
    layout = gen.paged_layout([40, 70], 32, gen.generator(21))
    case = gen.fused_case(22, layout, 3, Hq=4, Hkv=2)
    kc = np.full((layout.num_pages, 2, 32, 128), 0xA5, np.uint8)
    vc = kc.copy()
    q_out = oracle.qk_norm_rope_insert(
        gen.bf16_bits(case.q), gen.bf16_bits(case.k), gen.bf16_bits(case.v), case.positions.numpy(),
        gen.bf16_bits(case.q_norm_w), gen.bf16_bits(case.k_norm_w), case.eps, case.cos_sin.numpy(),
        case.slots.numpy(), 0.02, 0.01, kc, vc)
    qb, kb = gen.bf16_bits(case.q), gen.bf16_bits(case.k)
    table = case.cos_sin.numpy()
    k_rot = np.empty_like(kb)
    for t in range(kb.shape[0]):
        pos = int(case.positions[t])
        for h in range(4):
            assert np.array_equal(q_out[t, h], oracle.norm_rope_row(qb[t, h], gen.bf16_bits(case.q_norm_w),
                                                                  case.eps, table[pos]))
        for h in range(2):
            k_rot[t, h] = oracle.norm_rope_row(kb[t, h], gen.bf16_bits(case.k_norm_w), case.eps, table[pos])
    kc2 = np.full_like(kc, 0xA5)
    vc2 = np.full_like(vc, 0xA5)
    oracle.cache_insert(k_rot, gen.bf16_bits(case.v), case.slots.numpy(), 0.02, 0.01, kc2, vc2)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


# -------------------------------------------------------------- attention

def _small_cache(seed, seq_lens, M, ps=4, Hq=4, Hkv=2, D=128, window=None, k_scale=0.02, v_scale=0.03):
    case = gen.layer_case(seed, seq_lens, M, ps, window=window, Hq=Hq, Hkv=Hkv, D=D)
    P = case.layout.num_pages
    kc = np.full((P, Hkv, ps, D), 0xA5, np.uint8)
    vc = np.full((P, Hkv, ps, D), 0xA5, np.uint8)
    for kk, vv, ss in ((case.k_prior, case.v_prior, case.slots_prior), (case.k_new, case.v_new, case.slots_new)):
        oracle.cache_insert(gen.bf16_bits(kk), gen.bf16_bits(vv), ss.numpy(), k_scale, v_scale, kc, vc)
    return case, kc, vc


# Both oracle implementations of the attention definition (the C loops and the
# numpy float64 one used at full workload sizes) answer to the same pins.
ATTN_IMPLS = {"c": oracle.paged_attention, "numpy": attention_np.paged_attention}


@pytest.fixture(params=sorted(ATTN_IMPLS))
def attn(request):
    return ATTN_IMPLS[request.param]


def _run(attn, case, kc, vc, k_scale=0.02, v_scale=0.03, window_left=None, **kw):
    wl = case.window_left if window_left is None else window_left
    return attn(gen.bf16_bits(case.q), kc, vc, case.layout.block_table.numpy(),
                                  case.layout.seq_lens.numpy(), k_scale, v_scale, case.sm_scale,
                                  window_left=wl, **kw)


def test_attention_worked_two_keys(attn):
    # q = e_0, key 0 = e_0 (code 1.0), key 1 = 0; V0 = 2.0 everywhere, V1 = 0.
    # sm_scale 1, scales 1: logits (1, 0) -> out = 2e/(1+e) in every dim.
    D = 128
    q = np.zeros((1, 1, 1, D), np.uint16)
    q[0, 0, 0, 0] = 0x3F80
    kc = np.zeros((1, 1, 2, D), np.uint8)
    vc = np.zeros((1, 1, 2, D), np.uint8)
    kc[0, 0, 0, 0] = 0x38
    vc[0, 0, 0, :] = 0x40
    out = attn(q, kc, vc, np.array([[0]], np.int32), np.array([2], np.int32),
                                 1.0, 1.0, 1.0)
    assert np.allclose(out, 2 * math.e / (1 + math.e), rtol=1e-15)


def test_attention_brute_force_hand_enumerated_masks(attn):
    # L = 6, M = 3: rows at positions 3, 4, 5.
    visible = {-1: [[0, 1, 2, 3], [0, 1, 2, 3, 4], [0, 1, 2, 3, 4, 5]],
               2: [[1, 2, 3], [2, 3, 4], [3, 4, 5]],
               0: [[3], [4], [5]]}
    case, kc, vc = _small_cache(31, [6], 3, ps=4, Hq=4, Hkv=2)
    qf = case.q.float().numpy().astype(np.float64)
    kd = oracle.e4m3_decode(kc) * 0.02
    vd = oracle.e4m3_decode(vc) * 0.03
    bt = case.layout.block_table.numpy()
    for wl, sets in visible.items():
        out = _run(attn, case, kc, vc, window_left=wl)
        for m in range(3):
            for h in range(4):
                hk = h // 2
                logits, vals = [], []
                for j in sets[m]:
                    page, off = bt[0, j // 4], j % 4
                    logits.append(sum(qf[0, m, h, d] * kd[page, hk, off, d] for d in range(128)) * case.sm_scale)
                    vals.append(vd[page, hk, off])
                mx = max(logits)
                wts = [math.exp(s - mx) for s in logits]
                ref = sum(wt * v for wt, v in zip(wts, vals)) / sum(wts)
                assert np.allclose(out[0, m, h], ref, rtol=1e-12, atol=1e-14)


def test_attention_constant_keys_give_mean_of_visible_values(attn):
    case, kc, vc = _small_cache(41, [37, 20], 5, ps=8, window=16)
    kc[:] = 0x3A                                   # every key equal
    out_sw = _run(attn, case, kc, vc)
    out_g = _run(attn, case, kc, vc, window_left=-1)
    vd = oracle.e4m3_decode(vc) * 0.03
    bt = case.layout.block_table.numpy()
    for b, L in enumerate([37, 20]):
        for m in range(5):
            p = L - 5 + m
            for h in range(4):
                for wl, out in ((15, out_sw), (-1, out_g)):
                    lo = 0 if wl < 0 else max(0, p - wl)
                    vals = [vd[bt[b, j // 8], h // 2, j % 8] for j in range(lo, p + 1)]
                    assert np.allclose(out[b, m, h], np.mean(vals, axis=0), rtol=1e-12, atol=1e-15)


def test_attention_single_key_returns_its_value(attn):
    case, kc, vc = _small_cache(51, [1], 1, ps=4)
    out = _run(attn, case, kc, vc)
    vd = oracle.e4m3_decode(vc) * 0.03
    page = case.layout.block_table[0, 0].item()
    for h in range(4):
        assert np.allclose(out[0, 0, h], vd[page, h // 2, 0], rtol=1e-15)


def test_attention_gqa_head_mapping(attn):
    case, kc, vc = _small_cache(61, [9], 2, ps=4, Hq=6, Hkv=3)
    for hk in range(3):
        vc[:, hk] = oracle.e4m3_encode(np.array([hk + 1.0], np.float32))[0]
    out = _run(attn, case, kc, vc, v_scale=1.0)
    for h in range(6):
        assert np.allclose(out[:, :, h], h // 2 + 1.0, rtol=1e-14)


def test_attention_page_permutation_invariance(attn):
    case, kc, vc = _small_cache(71, [30, 13], 3, ps=4, window=9)
    ref = _run(attn, case, kc, vc)
    rng = np.random.default_rng(0)
    perm = rng.permutation(kc.shape[0])             # new page i holds old page perm[i]
    inv = np.argsort(perm)
    bt = case.layout.block_table.numpy()
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    out = attn(gen.bf16_bits(case.q), np.ascontiguousarray(kc[perm]),
                                 np.ascontiguousarray(vc[perm]), bt2, case.layout.seq_lens.numpy(),
                                 0.02, 0.03, case.sm_scale, window_left=case.window_left)
    assert np.array_equal(out, ref)


def test_attention_equal_queries_in_group_give_equal_outputs(attn):
    case, kc, vc = _small_cache(81, [25], 4, ps=8, Hq=6, Hkv=2)
    case.q[:, :, 1] = case.q[:, :, 0]
    out = _run(attn, case, kc, vc)
    assert np.array_equal(out[:, :, 1], out[:, :, 0])
    assert not np.allclose(out[:, :, 3], out[:, :, 0])


def test_attention_short_sequence_sliding_equals_global(attn):
    case, kc, vc = _small_cache(91, [20, 7], 3, ps=4, window=20)
    assert np.array_equal(_run(attn, case, kc, vc), _run(attn, case, kc, vc, window_left=-1))
    case2, kc2, vc2 = _small_cache(91, [30], 3, ps=4, window=20)
    assert not np.allclose(_run(attn, case2, kc2, vc2), _run(attn, case2, kc2, vc2, window_left=-1))


def test_attention_split_combine_equals_unsplit():
    case, kc, vc = _small_cache(101, [45, 64], 4, ps=8, window=30)
    rows = np.array([(b, m, h) for b in range(2) for m in range(4) for h in range(4)], np.int32)
    args = (gen.bf16_bits(case.q), kc, vc, case.layout.block_table.numpy(), case.layout.seq_lens.numpy(),
            0.02, 0.03, case.sm_scale)
    ref = oracle.paged_attention_rows(*args, rows, window_left=case.window_left)
    for S in (1, 5, 8, 16, 100):
        out = oracle.paged_attention_rows(*args, rows, window_left=case.window_left, split_tokens=S)
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    full = _run(oracle.paged_attention, case, kc, vc)
    assert np.array_equal(ref.reshape(2, 4, 4, 128), full)


def test_attention_against_torch_sdpa_float64(attn):
    case, kc, vc = _small_cache(111, [33, 18], 5, ps=8, Hq=6, Hkv=2, window=12)
    out = _run(attn, case, kc, vc)
    kd = oracle.e4m3_decode(kc) * 0.02
    vd = oracle.e4m3_decode(vc) * 0.03
    bt = case.layout.block_table.numpy()
    qf = torch.from_numpy(case.q.float().numpy().astype(np.float64))
    for b, L in enumerate([33, 18]):
        keys = torch.from_numpy(np.stack([kd[bt[b, j // 8], :, j % 8] for j in range(L)], 1))
        vals = torch.from_numpy(np.stack([vd[bt[b, j // 8], :, j % 8] for j in range(L)], 1))
        keys = keys.repeat_interleave(3, dim=0)     # [Hq][L][D]
        vals = vals.repeat_interleave(3, dim=0)
        pos = torch.arange(L - 5, L)[:, None]
        j = torch.arange(L)[None, :]
        mask = (j <= pos) & (j >= pos - 11)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qf[b].transpose(0, 1), keys, vals, attn_mask=mask, scale=case.sm_scale)
        assert np.allclose(out[b], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_attention_prefill_from_empty_is_causal_sdpa(attn):
    """A whole sequence as new rows (L = M = 40, a prefill from an empty cache):
    row m sees keys 0..m, which is the textbook causal attention
    (scaled_dot_product_attention with is_causal=True, no hand-built mask)."""
    case, kc, vc = _small_cache(115, [40], 40, ps=8, Hq=6, Hkv=2)
    out = _run(attn, case, kc, vc)
    kd = oracle.e4m3_decode(kc) * 0.02
    vd = oracle.e4m3_decode(vc) * 0.03
    bt = case.layout.block_table.numpy()
    keys = torch.from_numpy(np.stack([kd[bt[0, j // 8], :, j % 8] for j in range(40)], 1)).repeat_interleave(3, 0)
    vals = torch.from_numpy(np.stack([vd[bt[0, j // 8], :, j % 8] for j in range(40)], 1)).repeat_interleave(3, 0)
    qf = torch.from_numpy(case.q.float().numpy().astype(np.float64))[0].transpose(0, 1)   # [Hq][M][D]
    ref = torch.nn.functional.scaled_dot_product_attention(qf, keys, vals, is_causal=True, scale=case.sm_scale)
    assert np.allclose(out[0], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_attention_prefill_chunk_constant_keys_running_mean(attn):
    """A chunk of M = 24 new rows at the end of L = 50 with every key equal:
    row m (position 26 + m) returns the mean of the values it sees -- all
    earlier positions (global) or the last W = 7 (window_left 6)."""
    case, kc, vc = _small_cache(117, [50], 24, ps=4, window=7)
    kc[:] = 0x3A
    vd = oracle.e4m3_decode(vc) * 0.03
    bt = case.layout.block_table.numpy()
    for wl in (6, -1):
        out = _run(attn, case, kc, vc, window_left=wl)
        for m in range(24):
            p = 26 + m
            lo = 0 if wl < 0 else max(0, p - wl)
            for h in range(4):
                vals = [vd[bt[0, j // 4], h // 2, j % 4] for j in range(lo, p + 1)]
                assert np.allclose(out[0, m, h], np.mean(vals, axis=0), rtol=1e-12, atol=1e-15)


def test_attention_bf16_cache_variant(attn):
    case = gen.layer_case(121, [19], 2, 4, Hq=4, Hkv=2)
    P = case.layout.num_pages
    kc = np.zeros((P, 2, 4, 128), np.uint16)
    vc = np.zeros((P, 2, 4, 128), np.uint16)
    for kk, vv, ss in ((case.k_prior, case.v_prior, case.slots_prior), (case.k_new, case.v_new, case.slots_new)):
        oracle.cache_insert(gen.bf16_bits(kk), gen.bf16_bits(vv), ss.numpy(), 1.0, 1.0, kc, vc,
                            cache_dtype=oracle.BF16)
    out = attn(gen.bf16_bits(case.q), kc, vc, case.layout.block_table.numpy(),
                                 case.layout.seq_lens.numpy(), 5.0, 7.0, case.sm_scale,
                                 cache_dtype=oracle.BF16)   # scales ignored for bf16
    kf = torch.cat([case.k_prior, case.k_new]).double()
    vf = torch.cat([case.v_prior, case.v_new]).double()
    qf = case.q.double()[0]                      # [M][Hq][D]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qf.transpose(0, 1), kf.transpose(0, 1).repeat_interleave(2, 0),
        vf.transpose(0, 1).repeat_interleave(2, 0),
        attn_mask=torch.arange(19)[None, :] <= torch.arange(17, 19)[:, None], scale=case.sm_scale)
    assert np.allclose(out[0], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_unvisited_pages_are_never_read(attn):
    case, kc, vc = _small_cache(131, [40], 3, ps=4, window=8)
    ref = _run(attn, case, kc, vc)
    bt = case.layout.block_table.clone()
    bt[0, :7] = -1                                   # keys 0..27 are outside every window
    out = attn(gen.bf16_bits(case.q), kc, vc, bt.numpy(), case.layout.seq_lens.numpy(),
                                 0.02, 0.03, case.sm_scale, window_left=7)
    assert np.array_equal(out, ref)
    bt[0, 9] = -1                                    # keys 36..39 are visible: must be rejected
    with pytest.raises(ValueError):
        attn(gen.bf16_bits(case.q), kc, vc, bt.numpy(), case.layout.seq_lens.numpy(),
                               0.02, 0.03, case.sm_scale, window_left=7)


@pytest.mark.parametrize("seq_lens,M,ps,window", [([300, 77], 12, 32, 100), ([130], 40, 64, None)])
def test_numpy_and_c_attention_agree(seq_lens, M, ps, window):
    """The two oracle implementations of one definition agree to float64
    rounding on a verifier-shaped layer (72/8 heads) and a prefill chunk."""
    case = gen.layer_case(141 + M, seq_lens, M, ps, window=window)
    P = case.layout.num_pages
    kc = np.full((P, 8, ps, 128), 0xA5, np.uint8)
    vc = kc.copy()
    for kk, vv, ss in ((case.k_prior, case.v_prior, case.slots_prior), (case.k_new, case.v_new, case.slots_new)):
        oracle.cache_insert(gen.bf16_bits(kk), gen.bf16_bits(vv), ss.numpy(), case.k_scale, case.v_scale, kc, vc)
    args = (gen.bf16_bits(case.q), kc, vc, case.layout.block_table.numpy(), case.layout.seq_lens.numpy(),
            case.k_scale, case.v_scale, case.sm_scale)
    a = oracle.paged_attention(*args, window_left=case.window_left)
    b = attention_np.paged_attention(*args, window_left=case.window_left)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------- per-head scales
# An extension the pages do not use (their checkpoint asks for one scale per
# tensor, "KV-cache precision decision", "What the official checkpoint
# requests"): KV head h is encoded and decoded with its own scale.  Pinned by
# reduction to the per-tensor routines pinned above, head by head, and by a
# closed form.

def _per_head_case(seed=151, seq_lens=(45, 20), M=5, ps=8, Hq=6, Hkv=3, window=None):
    case = gen.layer_case(seed, list(seq_lens), M, ps, window=window, Hq=Hq, Hkv=Hkv, k_head_scale=(0.25, 4.0))
    ks = np.array([0.011, 0.023, 0.047], np.float32)[:Hkv]
    vs = np.array([0.031, 0.0155, 0.062], np.float32)[:Hkv]
    return case, ks, vs


def _insert_all(case, insert, kc, vc, ks, vs):
    for kk, vv, ss in ((case.k_prior, case.v_prior, case.slots_prior), (case.k_new, case.v_new, case.slots_new)):
        insert(gen.bf16_bits(kk), gen.bf16_bits(vv), ss.numpy(), ks, vs, kc, vc)


def test_per_head_insert_reduces_to_per_tensor_per_head():
    case, ks, vs = _per_head_case()
    P, Hkv = case.layout.num_pages, 3
    kc = np.full((P, Hkv, 8, 128), 0xA5, np.uint8)
    vc = kc.copy()
    _insert_all(case, oracle.cache_insert_per_head, kc, vc, ks, vs)
    for h in range(Hkv):
        kt = np.full_like(kc, 0xA5)
        vt = kt.copy()
        _insert_all(case, oracle.cache_insert, kt, vt, float(ks[h]), float(vs[h]))
        assert np.array_equal(kc[:, h], kt[:, h]) and np.array_equal(vc[:, h], vt[:, h]), h
    # the heads' scales differ, so the heads' bytes must differ from a
    # single-scale insert somewhere (a scale index dropped would pass above
    # only for head 0)
    k0 = np.full_like(kc, 0xA5)
    v0 = k0.copy()
    _insert_all(case, oracle.cache_insert, k0, v0, float(ks[0]), float(vs[0]))
    assert not np.array_equal(kc[:, 1:], k0[:, 1:]) and not np.array_equal(vc[:, 1:], v0[:, 1:])


def test_per_head_insert_equal_scales_equal_per_tensor():
    case, _, _ = _per_head_case(seed=152)
    P = case.layout.num_pages
    kc = np.full((P, 3, 8, 128), 0xA5, np.uint8)
    vc = kc.copy()
    _insert_all(case, oracle.cache_insert_per_head, kc, vc, np.full(3, 0.02, np.float32), np.full(3, 0.03, np.float32))
    kt = np.full_like(kc, 0xA5)
    vt = kt.copy()
    _insert_all(case, oracle.cache_insert, kt, vt, 0.02, 0.03)
    assert np.array_equal(kc, kt) and np.array_equal(vc, vt)


PER_HEAD_ATTN = {"c": oracle.paged_attention_per_head, "numpy": attention_np.paged_attention}


@pytest.mark.parametrize("impl", sorted(PER_HEAD_ATTN))
@pytest.mark.parametrize("window", [None, 9])
def test_per_head_attention_reduces_to_per_tensor_per_head(impl, window):
    case, ks, vs = _per_head_case(seed=153, window=window)
    P, Hkv, G = case.layout.num_pages, 3, 2
    kc = np.full((P, Hkv, 8, 128), 0xA5, np.uint8)
    vc = kc.copy()
    _insert_all(case, oracle.cache_insert_per_head, kc, vc, ks, vs)
    q, bt, sl = gen.bf16_bits(case.q), case.layout.block_table.numpy(), case.layout.seq_lens.numpy()
    out = PER_HEAD_ATTN[impl](q, kc, vc, bt, sl, ks.astype(np.float64), vs.astype(np.float64), case.sm_scale,
                              window_left=case.window_left)
    for hk in range(Hkv):
        ref = oracle.paged_attention(q, kc, vc, bt, sl, float(ks[hk]), float(vs[hk]), case.sm_scale,
                                     window_left=case.window_left)
        assert np.allclose(out[:, :, hk * G:(hk + 1) * G], ref[:, :, hk * G:(hk + 1) * G], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("impl", sorted(PER_HEAD_ATTN))
def test_per_head_attention_constant_keys_closed_form(impl):
    """Equal keys in every head: each row returns v_scale[hk] times the mean
    of its visible V codes' values, for every head's own v_scale."""
    case, ks, vs = _per_head_case(seed=154)
    P, Hkv, G, M = case.layout.num_pages, 3, 2, 5
    kc = np.full((P, Hkv, 8, 128), 0x3A, np.uint8)
    vc = np.full((P, Hkv, 8, 128), 0xA5, np.uint8)
    _insert_all(case, oracle.cache_insert_per_head, np.empty_like(kc), vc, ks, vs)
    out = PER_HEAD_ATTN[impl](gen.bf16_bits(case.q), kc, vc, case.layout.block_table.numpy(),
                              case.layout.seq_lens.numpy(), ks.astype(np.float64), vs.astype(np.float64),
                              case.sm_scale)
    codes = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    bt = case.layout.block_table.numpy()
    for b, L in enumerate([45, 20]):
        for m in range(M):
            p = L - M + m
            for h in range(6):
                hk = h // G
                vals = [codes[vc[bt[b, j // 8], hk, j % 8]] for j in range(0, p + 1)]
                assert np.allclose(out[b, m, h], float(vs[hk]) * np.mean(vals, axis=0), rtol=1e-12, atol=1e-15)


def test_per_head_scales_of_the_generator():
    """minmax/448 of each head's whole K and V, fp32."""
    case, _, _ = _per_head_case(seed=155)
    k = torch.cat([case.k_prior, case.k_new]).float()
    v = torch.cat([case.v_prior, case.v_new]).float()
    for h in range(3):
        assert case.k_scale_h[h].item() == float(np.float32(k[:, h].abs().max().item()) / np.float32(448.0))
        assert case.v_scale_h[h].item() == float(np.float32(v[:, h].abs().max().item()) / np.float32(448.0))
    assert case.k_scale == float(case.k_scale_h.max()) and case.v_scale == float(case.v_scale_h.max())


def load_norm_rope_rounding():
    """The exact-arithmetic row of tests/golden/norm_rope_rounding.txt."""
    vals = {}
    for line in open(os.path.join(GOLDEN, "norm_rope_rounding.txt")):
        if line.strip() and not line.startswith("#"):
            key, *rest = line.split()
            vals[key] = rest
    hexes = lambda k, t: np.array([int(h, 16) for h in vals[k]], t)   # noqa: E731
    return dict(x=hexes("x", np.uint16), w=hexes("w", np.uint16), cs=hexes("cs", np.uint32).view(np.float32),
                out=hexes("out", np.uint16), eps=np.uint32(int(vals["eps"][0], 16)).view(np.float32),
                pos=int(vals["pos"][0]))


def test_norm_rope_rounding_sensitive_fixture():
    """A row whose output bits change if the bf16 rounding after the
    normalisation is dropped, if the 32 lane sums are added sequentially
    instead of pairwise, or if RoPE rounds its product before the fma: the
    oracle must reproduce the exact-arithmetic evaluation bit for bit."""
    f = load_norm_rope_rounding()
    assert f["eps"] == np.float32(1e-6)
    table = oracle.rope_table(1e6, f["pos"] + 1, 128)
    assert np.array_equal(table[f["pos"]], f["cs"])             # the stored row is the model's table row
    out = oracle.norm_rope_row(f["x"], f["w"], float(f["eps"]), f["cs"])
    assert np.array_equal(out, f["out"]), np.nonzero(out != f["out"])
