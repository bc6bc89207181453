"""The error path of the bounded device waits, on the GPU, without a fault or a
hang: a wait on an mbarrier that nothing completes gives up after its limit,
raises the timeout bit of the device status word, the CTA's other role leaves
on the abort flag, and the context stays usable for the next call."""
import time

import numpy as np
import pytest

from sparsified_long_context_gb300 import workloads as W

from gpu_harness import assert_close, bf16_tensor_to_f64, oracle_attention_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [2000, 50000])
def test_bounded_wait_gives_up_and_the_context_stays_usable(limit_us):
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import DeviceInputs, StepBuffers, run_attention
    B.unip_get_device_status(clear=True)
    res = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    B.unip_selftest_bounded_wait(limit_us, res)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    st = B.unip_get_device_status(clear=True)
    gave_up_a, gave_up_b, waited_b_us = res.cpu().tolist()
    assert st & 0x8, B.describe_status(st)                 # UNIP_DEV_TIMEOUT
    assert gave_up_a == 1 and gave_up_b == 1
    assert waited_b_us < 500000                            # left on the abort flag, not on its own 1 s limit
    assert waited_b_us >= limit_us * 0.5
    assert wall < 5.0
    # the context still runs a normal call correctly, with a clean status
    wl = W.tiny_packed()
    di = DeviceInputs.from_workload(wl, "cuda", with_hidden=False)
    bufs = StepBuffers(di)
    run_attention(di, bufs)
    torch.cuda.synchronize()
    assert B.unip_get_device_status(clear=True) == 0
    ref, _ = oracle_attention_rows(wl, None)
    assert_close(bf16_tensor_to_f64(bufs.out), ref, what="attention after the self-test")
