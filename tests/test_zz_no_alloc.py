"""qg_gemv_static_ws: the GEMV for callers that cannot allocate device memory where they
call it (for example a plugin whose host framework owns every device allocation), which
runs on the library's fixed device scratch array instead of a caller workspace.  Its
results must be bit-identical to qg_gemv with a workspace (same kernels, same plans); two
calls in a row on one stream share the array and must not disturb each other; problems
whose workspace would exceed the array are refused.  This file is collected last."""
import numpy as np
import pytest
import torch

import oracle
import synth
from qg_testlib import assert_within, dev, host, qg_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()

CASES = [
    (synth.Q4_K, 2048, 4096, 1),     # plain rows
    (synth.Q6_K, 300, 5120, 4),      # several tokens
    (synth.Q4_0, 5, 8192, 3),        # few rows: split-K partial sums live in the scratch too
    (synth.IQ4_XS, 64, 17408, 16),   # long rows at the largest batch
]


@pytest.mark.parametrize("fmt,N,K,M", CASES, ids=[f"{synth.FORMAT_NAMES[c[0]]}-{c[1]}x{c[2]}-M{c[3]}" for c in CASES])
def test_static_ws_two_calls_match_gemv(qg, fmt, N, K, M):
    assert qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, M, N, K) <= qg.QG_STATIC_WS_BYTES
    g = np.random.default_rng(N * 7 + K + M)
    W1, W2 = dev(synth.weights(fmt, N, K, g)), dev(synth.weights(fmt, N, K, g))
    x1, x2 = dev(synth.activations(M, K, g)), dev(synth.activations(M, K, g))
    s = torch.cuda.current_stream()
    # two calls in a row on one stream, then the workspace entry point
    y1 = qg.qg_gemv_static_ws(fmt, W1, x1, N, stream=s)
    y2 = qg.qg_gemv_static_ws(fmt, W2, x2, N, stream=s)
    r1 = qg.qg_gemv(fmt, W1, x1, N, stream=s)
    r2 = qg.qg_gemv(fmt, W2, x2, N, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(y1, r1)
    assert torch.equal(y2, r2)
    assert not torch.equal(y1, y2)
    assert qg.qg_device_error() == 0
    # and against the oracle, not only against the workspace entry point
    for W, x, y in ((W1, x1, y1), (W2, x2, y2)):
        Wn, xn = host(W), host(x)
        xq, xd, xs = oracle.quantize_act(xn)
        assert_within(host(y), oracle.gemv_q(fmt, Wn, xq, xd, xs, N, K), oracle.absdot(fmt, Wn, xq, xd, N, K),
                      "static-scratch gemv")


def test_static_ws_leftover_scratch_from_a_larger_call(qg):
    """A call that fills most of the scratch (split-K partial sums of 16 tokens) directly
    followed by a smaller split-K call: the second call reads only what it wrote itself."""
    big = (synth.Q4_0, 3, 131072 // 4, 16)
    small = (synth.Q4_0, 5, 8192, 3)
    need_big = qg.qg_workspace_size(qg.QG_OP_GEMV, big[0], big[3], big[1], big[2])
    need_small = qg.qg_workspace_size(qg.QG_OP_GEMV, small[0], small[3], small[1], small[2])
    assert need_small < need_big <= qg.QG_STATIC_WS_BYTES
    g = np.random.default_rng(2024)
    s = torch.cuda.current_stream()
    outs = []
    for fmt, N, K, M in (big, small, big, small):
        W, x = synth.weights(fmt, N, K, g), synth.activations(M, K, g)
        y = qg.qg_gemv_static_ws(fmt, dev(W), dev(x), N, stream=s)
        outs.append((fmt, N, K, W, x, y))
    torch.cuda.synchronize()
    for fmt, N, K, W, x, y in outs:
        xq, xd, xs = oracle.quantize_act(x)
        assert_within(host(y), oracle.gemv_q(fmt, W, xq, xd, xs, N, K), oracle.absdot(fmt, W, xq, xd, N, K),
                      f"static scratch {N}x{K} after a larger call")
    assert qg.qg_device_error() == 0


def test_static_ws_refuses_oversize(qg):
    fmt, N, K, M = synth.Q8_0, 1, 131072, 16
    need = qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, M, N, K)
    assert need > qg.QG_STATIC_WS_BYTES
    W = torch.zeros((N, synth.row_bytes(fmt, K)), dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), dtype=torch.float32, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.qg_gemv_static_ws(fmt, W, x, N)
    assert e.value.status == qg.QG_EWORKSPACE
