"""The failure path on the GPU, without a fault: a kernel's bounded wait on
a barrier that nothing arrives on gives up after its time limit, reports the
timeout in the device error word, and the context stays usable."""
import time

import pytest
import torch

from split_flash_decoding_gb300 import workloads as W
from tests.helpers import assert_close, oracle_result

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def attn():
    from split_flash_decoding_gb300 import build
    build.build()
    from split_flash_decoding_gb300 import attn as a
    a.attn_device_error_flags(clear=True)
    yield a
    a.attn_device_error_flags(clear=True)


def test_wait_timeout_is_reported_and_context_stays_usable(attn):
    assert attn.attn_device_error_flags(clear=True) == 0
    t0 = time.perf_counter()
    attn.attn_selftest_wait_timeout()
    flags = attn.attn_device_error_flags(clear=True)
    dt = time.perf_counter() - t0
    assert flags & 1, f"timeout bit not set (flags {flags:#x})"
    assert 0.2 < dt < 10.0, f"the wait gave up after {dt:.3f} s"
    # The context still works: a decode call right after matches the oracle.
    w = W.tiny_decode(device=DEV)
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=w.group,
                                scale=w.scale, max_kv_len=w.max_kv_len, num_partitions=3)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "decode after a timed-out wait")
    assert attn.attn_device_error_flags(clear=True) == 0
