"""GPU parity of the prefill GEMM on the tensor cores (qg_prefill_gemm) against the oracle's
fp16-operand reading ("01 · 阶段总览", section 九 and section 四 issue ⑮): the fp16 weights
the kernel multiplies are bit-exact (test hook qg_dequant_f16), and y is within the
per-element bound |y - y_ref| <= 1e-5 * sum_k |w16 x16| + 1e-6, the fp32 accumulation being
the only difference.  Shapes span several row tiles, token tiles and K-slices with ragged
tails (N, M and K not multiples of the tiles; K % 64 == 32 for 32-element blocks), and the
dense-27B FFN shapes at 512 tokens on sampled rows.  All calls go through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from qg_testlib import FMTS, FMT_IDS, assert_within, dev, host, qg_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_dequant_f16_bit_exact(qg, fmt):
    qk = synth.BLOCK_ELEMS[fmt]
    g = np.random.default_rng(4100 + fmt)
    for N, K in [(3, qk), (37, 3 * qk), (64, 4096)]:
        W = synth.weights(fmt, N, K, g)
        got = host(qg.qg_dequant_f16(fmt, dev(W), N, K)).view(np.uint16)
        np.testing.assert_array_equal(got, oracle.dequant_f16(fmt, W, N, K))


def _small_cases(qk):
    return [
        (300, max(1024, 4 * qk), 37),   # 3 row tiles (ragged), one token tile of 48
        (130, 3 * qk, 1),               # one token; K % 64 == 32 for 32-element blocks
        (129, 2 * max(qk, 128), 257),   # two token tiles, the second of one token
        (40, 8192, 300),                # one row tile, K split into slices
    ]


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_prefill_small_shapes(qg, fmt):
    qk = synth.BLOCK_ELEMS[fmt]
    g = np.random.default_rng(5200 + fmt)
    for N, K, M in _small_cases(qk):
        W = synth.weights(fmt, N, K, g)
        x = synth.activations(M, K, g)
        y = host(qg.qg_prefill_gemm(fmt, dev(W), dev(x), N))
        y_ref, sabs = oracle.prefill_gemm(fmt, W, x, N, K)
        assert_within(y, y_ref, sabs, f"prefill {synth.FORMAT_NAMES[fmt]} N={N} K={K} M={M}")
    assert qg.qg_device_error() == 0


FULL = [(synth.Q4_K, 17408, 5120), (synth.Q4_K, 5120, 17408), (synth.Q4_0, 17408, 5120), (synth.Q4_0, 5120, 17408)]


@pytest.mark.parametrize("fmt,N,K", FULL, ids=[f"{synth.FORMAT_NAMES[f]}-{n}x{k}" for f, n, k in FULL])
def test_prefill_full_size_sampled_rows(qg, fmt, N, K):
    M = 512
    g = np.random.default_rng(N + K + fmt)
    W = synth.weights(fmt, N, K, g)
    x = synth.activations(M, K, g)
    y = host(qg.qg_prefill_gemm(fmt, dev(W), dev(x), N))
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 129, N - 129, N - 128, N - 1], g.integers(0, N, 40)]))
    rb = synth.row_bytes(fmt, K)
    Ws = np.ascontiguousarray(W.reshape(N, rb)[rows])
    y_ref, sabs = oracle.prefill_gemm(fmt, Ws, x, len(rows), K)
    assert_within(y[:, rows], y_ref, sabs, f"prefill {synth.FORMAT_NAMES[fmt]} {N}x{K} M={M}")
    assert qg.qg_device_error() == 0


def test_prefill_rejects_bad_arguments(qg):
    torch = pytest.importorskip("torch")
    W = torch.zeros((4, synth.row_bytes(synth.Q4_K, 256)), dtype=torch.uint8, device="cuda")
    x = torch.zeros((3, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.qg_prefill_gemm(synth.Q4_K, W, torch.zeros((3, 255), dtype=torch.float32, device="cuda"), 4)
    assert e.value.status == qg.QG_EINVAL
    with pytest.raises(qg.QGError) as e:
        qg.qg_prefill_gemm(synth.Q4_K, W, x, 4, ws=torch.zeros(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == qg.QG_EWORKSPACE


GROUPS = [(synth.Q4_K, 400), (synth.Q4_0, 600), (synth.Q6_K, 600)]


@pytest.mark.parametrize("fmt,M", GROUPS, ids=[f"{synth.FORMAT_NAMES[f]}-M{m}" for f, m in GROUPS])
def test_prefill_two_token_tiles_per_cta(qg, fmt, M):
    """Shapes whose plan gives every CTA two token tiles of 256 (two accumulators): M = 400
    (the second tile ragged) and M = 600 (the last CTA group holding one tile of 88)."""
    N, K = 17408, 1024
    g = np.random.default_rng(7000 + M + fmt)
    W = synth.weights(fmt, N, K, g)
    x = synth.activations(M, K, g)
    y = host(qg.qg_prefill_gemm(fmt, dev(W), dev(x), N))
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], g.integers(0, N, 28)]))
    rb = synth.row_bytes(fmt, K)
    y_ref, sabs = oracle.prefill_gemm(fmt, np.ascontiguousarray(W.reshape(N, rb)[rows]), x, len(rows), K)
    assert_within(y[:, rows], y_ref, sabs, f"prefill {synth.FORMAT_NAMES[fmt]} {N}x{K} M={M}")
    assert qg.qg_device_error() == 0
