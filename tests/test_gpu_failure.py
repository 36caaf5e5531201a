"""Failure detection on the device, without a GPU fault: a pipeline barrier
wait that by construction gets no arrival gives up after its limit, sets
FP8KV_DEV_WAIT_TIMEOUT in the device status word and returns; the host reads
the bit and the context keeps working (a real attention call afterwards is
still correct).  Nothing here traps, faults or hangs the GPU."""
import time

import pytest
import torch

from verify_attention_gb300 import build, inputs as gen
from tests.helpers import assert_close, gpu_attention, gpu_caches, oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    build.build()
    from verify_attention_gb300 import fp8kv as f
    f.fp8kv_device_status(clear=True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    f.fp8kv_selftest_bounded_wait(20000)                 # 20 ms
    status = f.fp8kv_device_status(clear=True)           # synchronises
    waited = time.perf_counter() - t0
    assert status & f.DEV_WAIT_TIMEOUT, hex(status)
    assert waited >= 0.019, waited
    assert f.fp8kv_device_status(clear=True) == 0        # cleared
    # the context is intact: an attention call afterwards matches the oracle
    case = gen.layer_case(9900, [600], 12, 32, window=None)
    kc, vc, ks, vs = gpu_caches(case)
    out = gpu_attention(case, kc, vc, ks, vs)
    okc, ovc = oracle_caches(case)
    assert_close(out, oracle_attention(case, okc, ovc), "after the timed-out wait")
    assert f.fp8kv_device_status(clear=True) == 0


def test_bounded_wait_limit_is_validated_on_the_host():
    build.build()
    from verify_attention_gb300 import fp8kv as f
    for bad in (0, 2000001):
        with pytest.raises(f.Fp8kvError):
            f.fp8kv_selftest_bounded_wait(bad)
