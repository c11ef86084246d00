"""Guard bands around every buffer the library writes ("01 · 阶段总览", section 四, issue ⑬:
a byte-offset bug once wrote four times past a buffer into the weights).  Each workspace,
output and MoE routing output is handed over as the middle of a larger allocation whose
4 KB on either side hold a byte pattern; after the call the pattern must be intact.  The
workspace is exactly qg_workspace_size bytes, so the split-K and K-slice partial sums, the
tile images and the MoE / FFN intermediates inside it are covered too."""
import numpy as np
import pytest

import synth
from qg_testlib import dev, qg_module

pytestmark = pytest.mark.gpu

G = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def qg():
    return qg_module()


class Guarded:
    """A buffer of nbytes in the middle of an allocation with G guard bytes on each side."""

    def __init__(self, nbytes, dtype=None, shape=None):
        import torch
        self.n = nbytes
        self.raw = torch.full((nbytes + 2 * G,), PATTERN, dtype=torch.uint8, device="cuda")
        self.buf = self.raw[G:G + nbytes]
        if dtype is not None:
            self.t = self.buf.view(dtype).view(shape)

    def intact(self):
        import torch
        torch.cuda.synchronize()
        head = self.raw[:G].cpu().numpy()
        tail = self.raw[G + self.n:].cpu().numpy()
        return bool((head == PATTERN).all() and (tail == PATTERN).all())


def _check(*bufs):
    for i, b in enumerate(bufs):
        assert b.intact(), f"guard band of buffer {i} overwritten"


GEMV = [(synth.Q4_K, 17408, 5120, 1), (synth.Q4_0, 5, 8192, 3), (synth.Q4_K, 5120, 17408, 16),
        (synth.Q6_K, 300, 5120, 4), (synth.IQ4_XS, 64, 17408, 16), (synth.Q5_K, 4096, 4096, 1)]


@pytest.mark.parametrize("fmt,N,K,M", GEMV, ids=[f"{synth.FORMAT_NAMES[c[0]]}-{c[1]}x{c[2]}-M{c[3]}" for c in GEMV])
def test_gemv_guard_bands(qg, fmt, N, K, M):
    import torch
    g = np.random.default_rng(N + K + M)
    W = dev(synth.weights(fmt, N, K, g))
    x = dev(synth.activations(M, K, g))
    ws = Guarded(qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, M, N, K))
    y = Guarded(4 * M * N, torch.float32, (M, N))
    qg.qg_gemv(fmt, W, x, N, y=y.t, ws=ws.buf)
    _check(ws, y)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_ffn_guard_bands(qg, M):
    import torch
    fmt, H, I = synth.Q4_K, 1024, 2048
    g = np.random.default_rng(50 + M)
    Wg, Wu, Wd = dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, H, I, g))
    x = dev(synth.activations(M, H, g))
    ws = Guarded(qg.qg_workspace_size(qg.QG_OP_FFN_SUBLAYER, fmt, M, H, H, 0, 0, I))
    y = Guarded(4 * M * H, torch.float32, (M, H))
    qg.qg_ffn_sublayer(fmt, Wg, Wu, Wd, x, I, y=y.t, ws=ws.buf)
    _check(ws, y)


@pytest.mark.parametrize("s16", [False, True], ids=["int8", "s16"])
@pytest.mark.parametrize("M", [1, 4])
def test_moe_guard_bands(qg, M, s16):
    import torch
    fmt, H, E, topk, I = synth.Q4_K, 512, 16, 4, 256
    g = np.random.default_rng(60 + M)
    Wg, Wu = dev(synth.stacked_experts(fmt, E, I, H, g)), dev(synth.stacked_experts(fmt, E, I, H, g))
    Wd = dev(synth.stacked_experts(fmt, E, H, I, g))
    sg, su, sd = dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, I, H, g)), dev(synth.weights(fmt, H, I, g))
    Wr = dev(synth.router_weights(E, H, g))
    x = dev(synth.activations(M, H, g))
    op, call = (qg.QG_OP_MOE_FFN_S16, qg.qg_moe_ffn_s16) if s16 else (qg.QG_OP_MOE_FFN, qg.qg_moe_ffn)
    ws = Guarded(qg.qg_workspace_size(op, fmt, M, H, H, E, topk, I))
    y = Guarded(4 * M * H, torch.float32, (M, H))
    ids = Guarded(4 * M * topk, torch.int32, (M, topk))
    wts = Guarded(4 * M * topk, torch.float32, (M, topk))
    call(fmt, x, Wr, topk, Wg, Wu, Wd, sg, su, sd, I, y=y.t, topk_ids=ids.t, topk_w=wts.t, ws=ws.buf)
    _check(ws, y, ids, wts)


@pytest.mark.parametrize("N,K,M", [(40, 8192, 300), (300, 1024, 37), (17408, 1024, 600)])
def test_prefill_guard_bands(qg, N, K, M):
    import torch
    fmt = synth.Q4_K
    g = np.random.default_rng(N + M)
    W = dev(synth.weights(fmt, N, K, g))
    x = dev(synth.activations(M, K, g))
    ws = Guarded(qg.qg_workspace_size(qg.QG_OP_PREFILL, fmt, M, N, K))
    y = Guarded(4 * M * N, torch.float32, (M, N))
    qg.qg_prefill_gemm(fmt, W, x, N, y=y.t, ws=ws.buf)
    _check(ws, y)


def test_quantize_act_guard_bands(qg):
    import torch
    M, K = 3, 4096
    x = dev(synth.activations(M, K, np.random.default_rng(3)))
    xq = Guarded(M * K, torch.int8, (M, K))
    xd = Guarded(4 * M * K // 32, torch.float32, (M, K // 32))
    xs = Guarded(4 * M * K // 32, torch.int32, (M, K // 32))
    qg.qg_quantize_act(x, xq.t, xd.t, xs.t)
    _check(xq, xd, xs)


def test_no_device_error_recorded(qg):
    assert qg.qg_device_error() == 0
