"""The calls capture into CUDA graphs: every op of the path (GEMV with one and with several
tokens, FFN sublayer, MoE FFN with int8 and with s16 activations, prefill GEMM) is recorded
once on a capture stream, its inputs are then overwritten in place and the graph replayed.
Each replay is checked against the oracle on the new inputs (the GEMV and the prefill GEMM
directly; the FFN sublayer and the MoE stage by stage, from the intermediates the replay
left in the workspace, with the contracts of the direct-call tests), and equals a direct
call on the same inputs bit for bit (the kernels are deterministic and allocate nothing, so
a captured chain of preparation and engine launches, with their programmatic dependent
launches, replays exactly)."""
import numpy as np
import pytest

import oracle
import synth
from qg_testlib import assert_within, dev, host, qg_module
from test_gpu_moe_ffn import _check_moe, _ws_view
from test_gpu_moe_s16 import _check_moe16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()


def _replays(fn, inputs, fresh, outputs, check):
    """Capture fn() on a side stream, then for each set of fresh input arrays: copy them
    into the captured input tensors, replay, check the outputs against the oracle
    (check(arrays)), and compare them with a direct call."""
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
        check(arrays)
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
    Wn = synth.weights(fmt, N, K, g)
    W = dev(Wn)
    x = dev(synth.activations(M, K, g))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, M, N, K), 16), dtype=torch.uint8, device="cuda")
    fresh = [[synth.activations(M, K, g)] for _ in range(2)]

    def check(arrays):
        xq, xd, xs = oracle.quantize_act(arrays[0])
        assert_within(host(y), oracle.gemv_q(fmt, Wn, xq, xd, xs, N, K), oracle.absdot(fmt, Wn, xq, xd, N, K),
                      "gemv replay")

    _replays(lambda s: qg.qg_gemv(fmt, W, x, N, y=y, ws=ws, stream=s), [x], fresh, [y], check)


@pytest.mark.parametrize("fmt,N,K", [(synth.Q4_K, 2048, 4096), (synth.Q4_0, 1000, 2048)])
def test_gemv_first_call_inside_capture(qg, fmt, N, K):
    """A one-token call made first inside a stream capture, on buffers just allocated (64 MB
    of fresh device memory, so that the activations' memory-type query of the call most
    likely runs during the capture): the replay must be within bound of the oracle."""
    import torch
    g = np.random.default_rng(51 + K)
    Wn = synth.weights(fmt, N, K, g)
    W = dev(Wn)
    fresh = torch.empty(16 << 20, dtype=torch.float32, device="cuda")
    x = fresh[(8 << 20):(8 << 20) + K].view(1, K)
    x.copy_(dev(synth.activations(1, K, g)))
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, 1, N, K), 16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(gr, stream=s):
            qg.qg_gemv(fmt, W, x, N, y=y, ws=ws, stream=s)
    gr.replay()
    torch.cuda.synchronize()
    xq, xd, xs = oracle.quantize_act(host(x))
    assert_within(host(y), oracle.gemv_q(fmt, Wn, xq, xd, xs, N, K), oracle.absdot(fmt, Wn, xq, xd, N, K),
                  "first call captured")


@pytest.mark.parametrize("M", [1, 2])
def test_ffn_graph_replay(qg, M):
    import torch
    fmt, H, I = synth.Q4_K, 1024, 2048
    g = np.random.default_rng(21 + M)
    Wgn, Wun, Wdn = synth.weights(fmt, I, H, g), synth.weights(fmt, I, H, g), synth.weights(fmt, H, I, g)
    Wg, Wu, Wd = dev(Wgn), dev(Wun), dev(Wdn)
    x = dev(synth.activations(M, H, g))
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    nws = qg.qg_workspace_size(qg.QG_OP_FFN_SUBLAYER, fmt, M, H, H, 0, 0, I)
    ws = torch.zeros(max(nws, 16), dtype=torch.uint8, device="cuda")
    off = qg.qg_ffn_ws_layout(fmt, M, H, I)
    fresh = [[synth.activations(M, H, g)] for _ in range(2)]

    def check(arrays):
        # stage by stage: g, u against the oracle; y against the oracle's down projection
        # of the GPU's own h, requantized by the oracle
        xq, xd, xs = oracle.quantize_act(arrays[0])
        gg = _ws_view(ws, off[0], M * I, np.float32).reshape(M, I)
        uu = _ws_view(ws, off[1], M * I, np.float32).reshape(M, I)
        hh = _ws_view(ws, off[2], M * I, np.float32).reshape(M, I)
        assert_within(gg, oracle.gemv_q(fmt, Wgn, xq, xd, xs, I, H), oracle.absdot(fmt, Wgn, xq, xd, I, H), "g")
        assert_within(uu, oracle.gemv_q(fmt, Wun, xq, xd, xs, I, H), oracle.absdot(fmt, Wun, xq, xd, I, H), "u")
        hq, hd, hs = oracle.requant(hh.astype(np.float64))
        assert_within(host(y), oracle.gemv_q(fmt, Wdn, hq, hd, hs, H, I), oracle.absdot(fmt, Wdn, hq, hd, H, I),
                      "ffn y replay")

    _replays(lambda s: qg.qg_ffn_sublayer(fmt, Wg, Wu, Wd, x, I, y=y, ws=ws, stream=s), [x], fresh, [y], check)


@pytest.mark.parametrize("s16", [False, True], ids=["int8", "s16"])
@pytest.mark.parametrize("M", [1, 3])
def test_moe_graph_replay(qg, M, s16):
    import torch
    fmt, H, E, topk, I = synth.Q4_K, 512, 16, 4, 256
    S = topk + 1
    g = np.random.default_rng(31 + M)
    inp = dict(Wg=synth.stacked_experts(fmt, E, I, H, g), Wu=synth.stacked_experts(fmt, E, I, H, g),
               Wd=synth.stacked_experts(fmt, E, H, I, g), sg=synth.weights(fmt, I, H, g),
               su=synth.weights(fmt, I, H, g), sd=synth.weights(fmt, H, I, g), Wr=synth.router_weights(E, H, g))
    W = {k: dev(v) for k, v in inp.items()}
    x = dev(synth.activations(M, H, g))
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((M, topk), dtype=torch.int32, device="cuda")
    wts = torch.empty((M, topk), dtype=torch.float32, device="cuda")
    op, call = (qg.QG_OP_MOE_FFN_S16, qg.qg_moe_ffn_s16) if s16 else (qg.QG_OP_MOE_FFN, qg.qg_moe_ffn)
    nws = qg.qg_workspace_size(op, fmt, M, H, H, E, topk, I)
    ws = torch.zeros(max(nws, 16), dtype=torch.uint8, device="cuda")
    off = (qg.qg_moe_s16_ws_layout if s16 else qg.qg_moe_ws_layout)(M, H, E, topk, I)
    fresh = [[synth.activations(M, H, g)] for _ in range(2)]

    def check(arrays):
        out = dict(y=host(y), ids=host(ids), w=host(wts),
                   h=_ws_view(ws, off[2], M * S * I, np.float32).reshape(M, S, I),
                   hd=_ws_view(ws, off[4], M * S * I // 32, np.float32).reshape(M * S, I // 32),
                   hs=_ws_view(ws, off[5], M * S * I // 32, np.int32).reshape(M * S, I // 32),
                   logits=_ws_view(ws, off[6], M * E, np.float32).reshape(M, E))
        if s16:
            gp = _ws_view(ws, off[0], M * S * 2 * I, np.float32).reshape(M, S, 2, I)
            up = _ws_view(ws, off[1], M * S * 2 * I, np.float32).reshape(M, S, 2, I)
            out.update(g=(gp[:, :, 0] + gp[:, :, 1]).astype(np.float32), u=(up[:, :, 0] + up[:, :, 1]).astype(np.float32),
                       hq=_ws_view(ws, off[3], M * S * I, np.int16).reshape(M * S, I))
            _check_moe16(fmt, dict(inp, x=arrays[0]), out, M, H, E, topk, I)
        else:
            out.update(g=_ws_view(ws, off[0], M * S * I, np.float32).reshape(M, S, I),
                       u=_ws_view(ws, off[1], M * S * I, np.float32).reshape(M, S, I),
                       hq=_ws_view(ws, off[3], M * S * I, np.int8).reshape(M * S, I))
            _check_moe(fmt, dict(inp, x=arrays[0]), out, M, H, E, topk, I)

    _replays(lambda s: call(fmt, x, W["Wr"], topk, W["Wg"], W["Wu"], W["Wd"], W["sg"], W["su"], W["sd"], I, y=y,
                            topk_ids=ids, topk_w=wts, ws=ws, stream=s),
             [x], fresh, [y, ids, wts], check)


@pytest.mark.parametrize("fmt,M", [(synth.Q4_K, 300), (synth.Q4_0, 600)])
def test_prefill_graph_replay(qg, fmt, M):
    import torch
    g = np.random.default_rng(41 + M)
    N, K = 1024, 2048
    Wn = synth.weights(fmt, N, K, g)
    W = dev(Wn)
    x = dev(synth.activations(M, K, g))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(qg.qg_workspace_size(qg.QG_OP_PREFILL, fmt, M, N, K), dtype=torch.uint8, device="cuda")
    fresh = [[synth.activations(M, K, g)] for _ in range(2)]

    def check(arrays):
        y_ref, sabs = oracle.prefill_gemm(fmt, Wn, arrays[0], N, K)
        assert_within(host(y), y_ref, sabs, "prefill replay")

    _replays(lambda s: qg.qg_prefill_gemm(fmt, W, x, N, y=y, ws=ws, stream=s), [x], fresh, [y], check)
