"""Failure detection without a GPU fault: every wait in the kernels is bounded, and a wait
that gives up sets the device error word instead of hanging ("01 · 阶段总览", section 二 ⑤:
an explicit warning instead of silent degradation).  The test hook runs the kernels' own
bounded wait on an mbarrier that nothing ever arrives at, with a short limit: the kernel
must return, the error word must read 1 (a bounded wait gave up) and be clear once read,
and the context must stay usable (a GEMV afterwards is exact and reports no error)."""
import time

import numpy as np
import pytest

import oracle
import synth
from qg_testlib import assert_within, dev, host, qg_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()


@pytest.mark.parametrize("limit_us", [100, 2000])
def test_bounded_wait_expires_and_reports(qg, limit_us):
    torch = pytest.importorskip("torch")
    assert qg.qg_device_error() == 0
    t0 = time.perf_counter()
    qg.qg_test_wait_expiry(limit_us * 1000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0, f"the wait did not give up in time ({elapsed:.3f} s)"
    assert qg.qg_device_error() == 1
    assert qg.qg_device_error() == 0  # read and cleared
    # the context is still usable: a GEMV right after is correct and clean
    fmt, N, K = synth.Q4_K, 256, 2048
    g = np.random.default_rng(limit_us)
    W, x = synth.weights(fmt, N, K, g), synth.activations(1, K, g)
    y = host(qg.qg_gemv(fmt, dev(W), dev(x), N))
    xq, xd, xs = oracle.quantize_act(x)
    assert_within(y, oracle.gemv_q(fmt, W, xq, xd, xs, N, K), oracle.absdot(fmt, W, xq, xd, N, K), "gemv after")
    assert qg.qg_device_error() == 0


def test_wait_expiry_rejects_bad_limits(qg):
    with pytest.raises(qg.QGError) as e:
        qg.qg_test_wait_expiry(10)
    assert e.value.status == qg.QG_EINVAL
