"""The calls capture into CUDA graphs: every op of the path (GEMV with one and with several
tokens, FFN sublayer, MoE FFN with int8 and with s16 activations) is recorded once on a
capture stream, its inputs are then overwritten in place and the graph replayed, and each
replay equals a direct call on the
same inputs bit for bit (the kernels are deterministic and allocate nothing, so a captured
chain of preparation and engine launches, with their programmatic dependent launches,
replays exactly)."""
import numpy as np
import pytest

import synth
from qg_testlib import dev, host, qg_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()


def _replays_equal_direct(fn, inputs, fresh, outputs):
    """Capture fn() on a side stream, then for each set of fresh input arrays: copy them
    into the captured input tensors, replay, and compare the outputs with a direct call."""
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn(s)
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            fn(s)
    torch.cuda.synchronize()
    for arrays in fresh:
        for t, a in zip(inputs, arrays):
            t.copy_(dev(a))
        gr.replay()
        torch.cuda.synchronize()
        got = [host(o).copy() for o in outputs]
        with torch.cuda.stream(s):
            fn(s)
        torch.cuda.synchronize()
        for g_, o in zip(got, outputs):
            np.testing.assert_array_equal(g_, host(o))


@pytest.mark.parametrize("fmt,M", [(synth.Q4_K, 1), (synth.Q4_0, 1), (synth.Q4_K, 4), (synth.Q6_K, 2)])
def test_gemv_graph_replay(qg, fmt, M):
    import torch
    g = np.random.default_rng(11 + M + fmt)
    N, K = 1000, 4096
    W = dev(synth.weights(fmt, N, K, g))
    x = dev(synth.activations(M, K, g))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, M, N, K), 16), dtype=torch.uint8, device="cuda")
    fresh = [[synth.activations(M, K, g)] for _ in range(2)]
    _replays_equal_direct(lambda s: qg.qg_gemv(fmt, W, x, N, y=y, ws=ws, stream=s), [x], fresh, [y])


@pytest.mark.parametrize("M", [1, 2])
def test_ffn_graph_replay(qg, M):
    import torch
    fmt, H, I = synth.Q4_K, 1024, 2048
    g = np.random.default_rng(21 + M)
    Wg, Wu = dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, I, H, g))
    Wd = dev(synth.weights(fmt, H, I, g))
    x = dev(synth.activations(M, H, g))
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    nws = qg.qg_workspace_size(qg.QG_OP_FFN_SUBLAYER, fmt, M, H, H, 0, 0, I)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    fresh = [[synth.activations(M, H, g)] for _ in range(2)]
    _replays_equal_direct(lambda s: qg.qg_ffn_sublayer(fmt, Wg, Wu, Wd, x, I, y=y, ws=ws, stream=s), [x], fresh,
                          [y])


@pytest.mark.parametrize("s16", [False, True], ids=["int8", "s16"])
@pytest.mark.parametrize("M", [1, 3])
def test_moe_graph_replay(qg, M, s16):
    import torch
    fmt, H, E, topk, I = synth.Q4_K, 512, 16, 4, 256
    g = np.random.default_rng(31 + M)
    Wg, Wu = dev(synth.stacked_experts(fmt, E, I, H, g)), dev(synth.stacked_experts(fmt, E, I, H, g))
    Wd = dev(synth.stacked_experts(fmt, E, H, I, g))
    sg, su = dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, I, H, g))
    sd = dev(synth.weights(fmt, H, I, g))
    Wr = dev(synth.router_weights(E, H, g))
    x = dev(synth.activations(M, H, g))
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((M, topk), dtype=torch.int32, device="cuda")
    wts = torch.empty((M, topk), dtype=torch.float32, device="cuda")
    op, call = (qg.QG_OP_MOE_FFN_S16, qg.qg_moe_ffn_s16) if s16 else (qg.QG_OP_MOE_FFN, qg.qg_moe_ffn)
    nws = qg.qg_workspace_size(op, fmt, M, H, H, E, topk, I)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    fresh = [[synth.activations(M, H, g)] for _ in range(2)]
    _replays_equal_direct(
        lambda s: call(fmt, x, Wr, topk, Wg, Wu, Wd, sg, su, sd, I, y=y, topk_ids=ids, topk_w=wts, ws=ws, stream=s),
        [x], fresh, [y, ids, wts])
