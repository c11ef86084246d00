"""Activations and outputs in page-locked host memory: the kernels read x (or its quantized
form) and write y, the top-k and the quantized activations straight through the host link,
and every result equals, bit for bit, the same call on device buffers."""
import numpy as np
import pytest

import synth
from qg_testlib import dev, host, qg_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()


def _pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _sync():
    import torch
    torch.cuda.synchronize()


@pytest.mark.parametrize("fmt,N,K,M", [(synth.Q4_K, 4096, 5120, 1), (synth.Q4_0, 1000, 4096, 4),
                                       (synth.Q6_K, 24, 2048, 2), (synth.Q8_0, 3, 1024, 1)],
                         ids=["one-token", "row-pairs", "split-k", "tiny"])
def test_gemv_host_x_and_y(qg, fmt, N, K, M):
    g = np.random.default_rng(900 + M + fmt)
    W = dev(synth.weights(fmt, N, K, g))
    x = synth.activations(M, K, g)
    y_dev = host(qg.qg_gemv(fmt, W, dev(x), N))
    y_host = qg.qg_gemv(fmt, W, _pinned(x), N)
    _sync()
    assert y_host.is_pinned()
    np.testing.assert_array_equal(y_host.numpy(), y_dev)


def test_quantize_and_gemv_q_host(qg):
    fmt, N, K, M = synth.Q5_K, 512, 2048, 3
    g = np.random.default_rng(901)
    W = dev(synth.weights(fmt, N, K, g))
    x = synth.activations(M, K, g)
    q_dev = [host(t) for t in qg.qg_quantize_act(dev(x))]
    q_host = qg.qg_quantize_act(_pinned(x))
    _sync()
    for a, b in zip(q_host, q_dev):
        np.testing.assert_array_equal(a.numpy(), b)
    y_dev = host(qg.qg_gemv_q(fmt, W, *[dev(a) for a in q_dev], N))
    y_host = qg.qg_gemv_q(fmt, W, *q_host, N)
    _sync()
    np.testing.assert_array_equal(y_host.numpy(), y_dev)


@pytest.mark.parametrize("M", [1, 2])
def test_ffn_sublayer_host(qg, M):
    """At one token the device-memory call quantizes x inside the gate/up kernel and the
    host-memory call through the preparation kernel: the same y bit for bit."""
    fmt, H, I = synth.Q4_K, 1024, 2816
    g = np.random.default_rng(902 + M)
    Wg, Wu, Wd = (dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, I, H, g)),
                  dev(synth.weights(fmt, H, I, g)))
    x = synth.activations(M, H, g)
    y_dev = host(qg.qg_ffn_sublayer(fmt, Wg, Wu, Wd, dev(x), I))
    y_host = qg.qg_ffn_sublayer(fmt, Wg, Wu, Wd, _pinned(x), I)
    _sync()
    np.testing.assert_array_equal(y_host.numpy(), y_dev)


@pytest.mark.parametrize("s16", [False, True], ids=["int8", "s16"])
def test_moe_host(qg, s16):
    import torch
    fmt, M, H, E, topk, I = synth.Q4_K, 2, 512, 16, 4, 256
    g = np.random.default_rng(903)
    Wg, Wu = dev(synth.stacked_experts(fmt, E, I, H, g)), dev(synth.stacked_experts(fmt, E, I, H, g))
    Wd = dev(synth.stacked_experts(fmt, E, H, I, g))
    sg, su, sd = dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, H, I, g))
    Wr = dev(synth.router_weights(E, H, g))
    x = synth.activations(M, H, g)
    call = qg.qg_moe_ffn_s16 if s16 else qg.qg_moe_ffn
    ids_d = torch.empty((M, topk), dtype=torch.int32, device="cuda")
    w_d = torch.empty((M, topk), dtype=torch.float32, device="cuda")
    y_dev = host(call(fmt, dev(x), Wr, topk, Wg, Wu, Wd, sg, su, sd, I, topk_ids=ids_d, topk_w=w_d))
    ids_h = torch.empty((M, topk), dtype=torch.int32, pin_memory=True)
    w_h = torch.empty((M, topk), dtype=torch.float32, pin_memory=True)
    y_host = call(fmt, _pinned(x), Wr, topk, Wg, Wu, Wd, sg, su, sd, I, topk_ids=ids_h, topk_w=w_h)
    _sync()
    np.testing.assert_array_equal(y_host.numpy(), y_dev)
    np.testing.assert_array_equal(ids_h.numpy(), host(ids_d))
    np.testing.assert_array_equal(w_h.numpy(), host(w_d))


def test_weights_must_be_device_memory(qg):
    fmt, N, K = synth.Q4_K, 16, 256
    g = np.random.default_rng(904)
    W = _pinned(synth.weights(fmt, N, K, g))
    with pytest.raises(ValueError):
        qg.qg_gemv(fmt, W, dev(synth.activations(1, K, g)), N)
