"""GPU parity of the insert kernels against the oracle: bit-exact bytes.
Every call goes through the C ABI (libfp8kv.so)."""
import numpy as np
import pytest
import torch

import oracle
from verify_attention_gb300 import build, inputs as gen
from tests.helpers import POISON_E4M3, gpu_caches, oracle_caches

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


def test_encoder_exhaustive_all_fp32_bit_patterns():
    """All 2^32 fp32 bit patterns through the device encoder vs the oracle."""
    chunk = 1 << 28
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    for first in range(0, 1 << 32, chunk):
        fp8kv().fp8kv_e4m3_encode_bits(first, chunk, out)
        got = out.cpu().numpy()
        want = oracle.e4m3_encode_bits(first, chunk)
        if not np.array_equal(got, want):
            bad = np.nonzero(got != want)[0][:8]
            raise AssertionError(f"chunk {first:#x}: mismatch at bit patterns "
                                 f"{[hex(first + int(i)) for i in bad]} gpu {got[bad]} oracle {want[bad]}")


@pytest.mark.parametrize("ps", [32, 64])
@pytest.mark.parametrize("seq_lens,M", [([256], 1), ([4096], 12), ([5, 70, 33], 3)])
def test_insert_bit_exact(seq_lens, M, ps):
    case = gen.layer_case(7000 + len(seq_lens) + ps, seq_lens, M, ps, outlier_frac=0.01)
    kc, vc, _, _ = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)
    # slots never named keep the poison byte
    assert (okc == POISON_E4M3).any() or sum(seq_lens) % ps == 0


def test_insert_saturation_scale():
    """scale = minmax/448/4: the largest quarter of magnitudes saturates to +-448."""
    case = gen.layer_case(7100, [600], 4, 64)
    case.k_scale /= 4
    case.v_scale /= 4
    kc, vc, _, _ = gpu_caches(case)
    okc, ovc = oracle_caches(case)
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    assert (okc & 0x7F == 0x7E).sum() > 100


def test_insert_negative_slots_skipped_and_bf16_cache():
    case = gen.layer_case(7200, [90], 5, 32)
    case.slots_new[1] = -1
    case.slots_new[3] = -7
    kc, vc, _, _ = gpu_caches(case, cache_dtype="bf16")
    okc, ovc = oracle_caches(case, cache_dtype="bf16")
    assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), okc)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy().view(np.uint16), ovc)
    kc8, vc8, _, _ = gpu_caches(case)
    okc8, ovc8 = oracle_caches(case)
    assert np.array_equal(kc8.cpu().numpy(), okc8) and np.array_equal(vc8.cpu().numpy(), ovc8)


def test_insert_bad_slot_is_flagged_not_written():
    f = fp8kv()
    case = gen.layer_case(7300, [40], 2, 32)
    kc, vc, ks, vs = gpu_caches(case)
    before = kc.clone()
    bad = torch.tensor([kc.shape[0] * 32 + 5, 10 ** 9], dtype=torch.int64, device="cuda")
    f.fp8kv_device_status(clear=True)
    f.fp8kv_cache_insert(case.k_new.cuda(), case.v_new.cuda(), bad, ks, vs, kc, vc)
    assert f.fp8kv_device_status(clear=True) & f.DEV_BAD_SLOT
    assert torch.equal(kc, before)


def _fused_gpu(case, layout, k_scale, v_scale):
    f = fp8kv()
    shape = (layout.num_pages, case.k.shape[1], layout.page_size, 128)
    kc = torch.full(shape, POISON_E4M3, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    q_out = torch.empty_like(case.q, device="cuda")
    ks = torch.tensor([k_scale], dtype=torch.float32, device="cuda")
    vs = torch.tensor([v_scale], dtype=torch.float32, device="cuda")
    f.fp8kv_qk_norm_rope_insert(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.positions.cuda(),
                                case.q_norm_w.cuda(), case.k_norm_w.cuda(), case.eps, case.cos_sin.cuda(),
                                q_out, case.slots.cuda(), ks, vs, kc, vc)
    return q_out, kc, vc


def _fused_oracle(case, layout, k_scale, v_scale):
    shape = (layout.num_pages, case.k.shape[1], layout.page_size, 128)
    kc = np.full(shape, POISON_E4M3, np.uint8)
    vc = kc.copy()
    q_out = oracle.qk_norm_rope_insert(
        gen.bf16_bits(case.q), gen.bf16_bits(case.k), gen.bf16_bits(case.v), case.positions.numpy(),
        gen.bf16_bits(case.q_norm_w), gen.bf16_bits(case.k_norm_w), case.eps, case.cos_sin.numpy(),
        case.slots.numpy(), k_scale, v_scale, kc, vc)
    return q_out, kc, vc


@pytest.mark.parametrize("seq_lens,M,ps", [([300, 17, 1024], 12, 32), ([64], 1, 64)])
def test_fused_norm_rope_insert_bit_exact(seq_lens, M, ps):
    layout = gen.paged_layout(seq_lens, ps, gen.generator(7400))
    case = gen.fused_case(7401, layout, M)
    qg, kg, vg = _fused_gpu(case, layout, 0.011, 0.013)
    qo, ko, vo = _fused_oracle(case, layout, 0.011, 0.013)
    assert np.array_equal(qg.cpu().view(torch.int16).numpy().view(np.uint16), qo)
    assert np.array_equal(kg.cpu().numpy(), ko)
    assert np.array_equal(vg.cpu().numpy(), vo)


def test_fused_cfg5_full_size_bit_exact():
    """The serving mix: 64 sequences x 12 new tokens at their true offsets."""
    lens = gen.cfg5_seq_lens()
    layout = gen.paged_layout(lens, 32, gen.generator(1005 * 100))
    case = gen.fused_case(1005 * 100 + 1, layout, 12)
    qg, kg, vg = _fused_gpu(case, layout, 0.012, 0.011)
    qo, ko, vo = _fused_oracle(case, layout, 0.012, 0.011)
    assert np.array_equal(qg.cpu().view(torch.int16).numpy().view(np.uint16), qo)
    assert np.array_equal(kg.cpu().numpy(), ko)
    assert np.array_equal(vg.cpu().numpy(), vo)


def test_fused_bad_position_flagged():
    f = fp8kv()
    layout = gen.paged_layout([50], 32, gen.generator(7500))
    case = gen.fused_case(7501, layout, 2)
    case.positions[0] = case.cos_sin.shape[0] + 3
    f.fp8kv_device_status(clear=True)
    _fused_gpu(case, layout, 0.01, 0.01)
    assert f.fp8kv_device_status(clear=True) & f.DEV_BAD_POSITION


def test_fused_kernel_reproduces_the_exact_arithmetic_row():
    """The rounding-sensitive row of tests/golden/norm_rope_rounding.txt as a Q
    head and as a K head of one token at its position: the fused kernel's q_out
    bits equal the exact-arithmetic evaluation, and its K bytes equal the
    E4M3 encoding of that row."""
    from tests.test_oracle import load_norm_rope_rounding
    fx = load_norm_rope_rounding()
    f = fp8kv()
    pos = fx["pos"]
    table = torch.from_numpy(oracle.rope_table(1e6, pos + 1, 128)).cuda()
    bf = lambda a: torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)   # noqa: E731
    x = bf(fx["x"])
    q = x.view(1, 1, 128).repeat(1, 2, 1).cuda()
    k = x.view(1, 1, 128).cuda()
    v = torch.zeros_like(k)
    w = bf(fx["w"]).cuda()
    q_out = torch.empty_like(q)
    kc = torch.full((2, 1, 32, 128), POISON_E4M3, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    one = torch.ones(1, device="cuda")
    f.fp8kv_qk_norm_rope_insert(q, k, v, torch.tensor([pos], device="cuda"), w, w, float(fx["eps"]), table, q_out,
                                torch.tensor([37], device="cuda"), one, one, kc, vc)
    got = q_out.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got[0, 0], fx["out"]) and np.array_equal(got[0, 1], fx["out"])
    want_k = oracle.e4m3_encode(((fx["out"].astype(np.uint32) << 16).view(np.float32)))
    assert np.array_equal(kc[1, 0, 5].cpu().numpy(), want_k)
