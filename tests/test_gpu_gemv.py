"""GPU parity of the activation quantizer, the per-block integer sums and the GEMV
against the CPU oracle.  Every call goes through the C ABI (via the thin binding)."""
import numpy as np
import pytest

import oracle
import synth
from qg_testlib import FMTS, FMT_IDS, assert_within, dev, host, qg_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()


def _special_x(M, K, g):
    x = synth.activations(M, K, g)
    nb = K // 32
    if nb >= 6:
        x[0, 0:32] = 0.0                                          # all-zero block
        x[0, 32:64] *= np.float32(1e-30)                          # tiny scale
        x[0, 64:96] *= np.float32(1e30)                           # huge scale
        x[0, 96:128] = np.round(x[0, 96:128] * 20) / 2            # exact half ties
        x[0, 96] = 127.0                                          # ... with d = 1
        x[0, 128:160] = np.float32(1e-41)                         # subnormal inputs
        x[0, 160:192] = -x[0, 160:192] ** 2                       # one-signed block
    return x


# ----------------------------------------------------------------------------- activation quantization
@pytest.mark.parametrize("M,K", [(1, 32), (3, 4096), (16, 17408), (2, 96)])
def test_quantize_act_bit_exact(qg, M, K):
    g = np.random.default_rng(M * 100003 + K)
    x = _special_x(M, K, g)
    xq, xd, xs = qg.qg_quantize_act(dev(x))
    oq, od, os_ = oracle.quantize_act(x)
    np.testing.assert_array_equal(host(xq), oq)
    np.testing.assert_array_equal(host(xd).view(np.uint32), od.view(np.uint32))
    np.testing.assert_array_equal(host(xs), os_)


def _near_tie_x(K, g):
    """Blocks whose quotients v / d lie within a few 1e-7 of half-integers (and some exactly
    on them), besides the special blocks: the cases where rounding v / d needs the exact
    quotient."""
    x = _special_x(1, K, g)
    nb = K // 32
    for b in range(8, nb, 3):
        a = np.float32(abs(g.standard_normal()) * 10.0 ** g.uniform(-3, 3)) + np.float32(1e-3)
        d = np.float32(a / np.float32(127))
        k = g.integers(-126, 126, size=32)
        v = (k + 0.5) * np.float64(d) * (1 + g.uniform(-3e-7, 3e-7, size=32) * (b % 2))
        v[0] = a
        x[0, 32 * b:32 * b + 32] = v.astype(np.float32)
    return x


@pytest.mark.parametrize("fmt,N,K", [(synth.Q4_K, 17408, 5120), (synth.Q4_K, 3000, 8192), (synth.Q4_0, 2048, 8192),
                                     (synth.Q6_K, 4096, 4096), (synth.IQ4_XS, 1000, 4096), (synth.Q8_0, 300, 2048),
                                     (synth.Q4_K, 5120, 17408)])
def test_one_token_in_kernel_quantization(qg, fmt, N, K):
    """At one token with the activations in device memory (rows up to 8192) the one-token
    engine quantizes x in every CTA; with them in page-locked host memory (or longer rows) a
    preparation kernel does.  The two must
    give the same y bit for bit (same tiles, same deterministic sums), on blocks that take
    every branch of the quantization rule, and y must be within bound of the oracle."""
    import torch
    g = np.random.default_rng(4242 + K + fmt)
    Wn = synth.weights(fmt, N, K, g)
    W = dev(Wn)
    x = _near_tie_x(K, g)
    y_dev = host(qg.qg_gemv(fmt, W, dev(x), N))
    y_host = qg.qg_gemv(fmt, W, torch.from_numpy(x).pin_memory(), N)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y_dev, y_host.numpy())
    xq, xd, xs = oracle.quantize_act(x)
    assert_within(y_dev, oracle.gemv_q(fmt, Wn, xq, xd, xs, N, K), oracle.absdot(fmt, Wn, xq, xd, N, K), "fused y")


@pytest.mark.parametrize("fmt,N,K", [(synth.Q4_K, 2048, 5120), (synth.Q4_0, 1000, 4096)])
def test_activations_only_4_byte_aligned(qg, fmt, N, K):
    """Activations 4-byte but not 16-byte aligned (a view one element into a buffer) take the
    preparation kernel instead of the in-kernel quantization: the same y bit for bit as the
    16-byte-aligned call, within bound of the oracle."""
    import torch
    g = np.random.default_rng(4343 + K)
    Wn = synth.weights(fmt, N, K, g)
    W = dev(Wn)
    xn = synth.activations(1, K, g)
    buf = torch.zeros(K + 4, dtype=torch.float32, device="cuda")
    buf[1:K + 1] = dev(xn)[0]
    x_off = buf[1:K + 1].view(1, K)
    assert x_off.data_ptr() % 16 == 4
    y_off = host(qg.qg_gemv(fmt, W, x_off, N))
    y_al = host(qg.qg_gemv(fmt, W, dev(xn), N))
    np.testing.assert_array_equal(y_off, y_al)
    xq, xd, xs = oracle.quantize_act(xn)
    assert_within(y_off, oracle.gemv_q(fmt, Wn, xq, xd, xs, N, K), oracle.absdot(fmt, Wn, xq, xd, N, K), "4-byte x")


# ----------------------------------------------------------------------------- integer contract
@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_block_dots_bit_exact(qg, fmt):
    qk = synth.BLOCK_ELEMS[fmt]
    g = np.random.default_rng(77 + fmt)
    for N, K, M in [(5, qk, 1), (37, 3 * qk, 3), (64, 4096, 2), (3, 17408, 1)]:
        W = synth.weights(fmt, N, K, g)
        x = _special_x(M, K, g)
        oq, od, os_ = oracle.quantize_act(x)
        dots, aux = qg.qg_block_dots(fmt, dev(W), dev(oq), dev(os_), N)
        want_d, want_a = oracle.block_dots(fmt, W, oq, os_, N, K)
        np.testing.assert_array_equal(host(dots), want_d)
        np.testing.assert_array_equal(host(aux), want_a)


# ----------------------------------------------------------------------------- GEMV element-wise
def _cases(qk):
    if qk == 32:
        Ks = [32, 96, 544, 1056, 5120]
    else:
        Ks = [256, 512, 768, 2304, 4096]
    out = []
    for i, K in enumerate(Ks):
        for N in (1, 7, 300, 1000):
            out.append((N, K, [1, 3, 8, 2, 16][(i + N) % 5]))
    return out


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_gemv_matches_oracle(qg, fmt):
    g = np.random.default_rng(1000 + fmt)
    worst = 0.0
    for N, K, M in _cases(synth.BLOCK_ELEMS[fmt]):
        W = synth.weights(fmt, N, K, g)
        x = _special_x(M, K, g)
        y = host(qg.qg_gemv(fmt, dev(W), dev(x), N))
        oq, od, os_ = oracle.quantize_act(x)
        y_ref = oracle.gemv_q(fmt, W, oq, od, os_, N, K)
        sabs = oracle.absdot(fmt, W, oq, od, N, K)
        worst = max(worst, assert_within(y, y_ref, sabs, f"gemv N={N} K={K} M={M}"))
    print(f"worst err/bound {worst:.3f}")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_gemv_q_prequantized_matches_oracle(qg, fmt):
    g = np.random.default_rng(2000 + fmt)
    for N, K, M in [(300, 4096, 1), (64, 4096, 5), (2, 2048, 16)]:
        W = synth.weights(fmt, N, K, g)
        x = synth.activations(M, K, g)
        oq, od, os_ = oracle.quantize_act(x)
        y = host(qg.qg_gemv_q(fmt, dev(W), dev(oq), dev(od), dev(os_), N))
        assert_within(y, oracle.gemv_q(fmt, W, oq, od, os_, N, K), oracle.absdot(fmt, W, oq, od, N, K),
                      f"gemv_q N={N} M={M}")


@pytest.mark.parametrize("fmt,N,K,M", [
    (synth.Q8_0, 20, 32768, 2),      # rows larger than a ring slot: K split into segments
    (synth.Q6_K, 50, 17408, 1),      # 14280-byte rows that start 8-byte aligned
    (synth.Q4_K, 300, 8192, 16),     # 16 tokens of activation tiles exceed one CTA: split along K
    (synth.IQ4_XS, 3, 65536, 4),     # split-K over many slices + segments
    (synth.Q4_0, 4099, 96, 1),       # tiny rows packed 8 per warp step, odd N
    (synth.Q4_0, 1037, 512, 1),      # one token: one 16-block task per row (two swapped halves)
    (synth.Q4_0, 333, 2560, 1),      # one token: 5 tasks of 16 blocks per row, rows wrap in a step
    (synth.Q4_0, 333, 2560, 2),      # two tokens on the same rows: 8-block tasks
    (synth.Q2_K, 77, 768, 1),        # odd superblocks per row: one-superblock tasks, 4-byte aligned
    (synth.Q3_K, 301, 2304, 3),      # 110-byte superblocks that start 2-byte aligned
    (synth.Q2_K, 5, 65536, 16),      # split-K with 16 tokens
])
def test_gemv_layout_paths(qg, fmt, N, K, M):
    g = np.random.default_rng(N + K + M)
    W = synth.weights(fmt, N, K, g)
    x = synth.activations(M, K, g)
    y = host(qg.qg_gemv(fmt, dev(W), dev(x), N))
    oq, od, os_ = oracle.quantize_act(x)
    assert_within(y, oracle.gemv_q(fmt, W, oq, od, os_, N, K), oracle.absdot(fmt, W, oq, od, N, K),
                  f"{synth.FORMAT_NAMES[fmt]} N={N} K={K} M={M}")


# ----------------------------------------------------------------------------- row pairs
# Two or more tokens on an un-split GEMV take the row-pair engine (two rows per task) for
# Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, IQ4_NL, Q4_K, Q5_K, Q6_K and IQ4_XS: odd row counts (the
# last pair has one row), stages that start and end inside a pair, and 2..16 tokens.
PAIR_CASES = [(fmt, N, K, M)
              for fmt, K in [(synth.Q4_K, 1280), (synth.Q4_0, 768), (synth.Q8_0, 384), (synth.Q5_1, 640),
                             (synth.Q6_K, 2304), (synth.Q5_K, 512), (synth.IQ4_XS, 1024), (synth.IQ4_NL, 1536)]
              for N, M in [(77, 2), (153, 3), (1001, 5), (2, 16)]]
# rows too long for the tiles of every token: row pairs over token chunks (the last chunk
# ragged), and 16 tokens per lane with the unit-outer Q4_K decode
PAIR_CASES += [(synth.Q4_K, 301, 17408, 8), (synth.Q4_K, 300, 17408, 15), (synth.Q4_0, 77, 17408, 6),
               (synth.Q6_K, 200, 17408, 16), (synth.Q8_0, 100, 8192, 16), (synth.Q4_K, 999, 2048, 16)]


@pytest.mark.parametrize("fmt,N,K,M", PAIR_CASES,
                         ids=[f"{synth.FORMAT_NAMES[f]}-{n}x{k}-M{m}" for f, n, k, m in PAIR_CASES])
def test_gemv_row_pairs(qg, fmt, N, K, M):
    g = np.random.default_rng(7000 + N + K + M + fmt)
    W = synth.weights(fmt, N, K, g)
    x = synth.activations(M, K, g)
    y = host(qg.qg_gemv(fmt, dev(W), dev(x), N))
    oq, od, os_ = oracle.quantize_act(x)
    assert_within(y, oracle.gemv_q(fmt, W, oq, od, os_, N, K), oracle.absdot(fmt, W, oq, od, N, K),
                  f"{synth.FORMAT_NAMES[fmt]} pairs N={N} K={K} M={M}")


# ----------------------------------------------------------------------------- full sizes, sampled rows
FULL = [
    (synth.Q8_0, 1024, 1024),
    (synth.Q4_0, 17408, 5120), (synth.Q4_0, 5120, 17408),
    (synth.Q4_K, 17408, 5120), (synth.Q4_K, 5120, 17408),
    (synth.Q5_K, 4096, 4096), (synth.Q6_K, 4096, 4096), (synth.IQ4_XS, 4096, 4096),
    (synth.Q6_K, 17408, 5120), (synth.Q6_K, 5120, 17408),
    (synth.Q4_1, 4096, 4096), (synth.Q5_0, 4096, 4096), (synth.Q5_1, 4096, 4096), (synth.IQ4_NL, 4096, 4096),
    (synth.Q2_K, 4096, 4096), (synth.Q3_K, 4096, 4096), (synth.Q2_K, 17408, 5120), (synth.Q3_K, 5120, 17408),
    # one-token tasks of 8 blocks (Q4_1, Q5_0, Q5_1, Q8_0) and 16 blocks (IQ4_NL), and
    # 110-byte Q3_K superblocks on the one-token engine (rows of 2200 bytes: 2-row groups)
    (synth.Q4_1, 17408, 5120), (synth.Q5_0, 5120, 17408), (synth.Q5_1, 17408, 5120),
    (synth.Q8_0, 17408, 5120), (synth.IQ4_NL, 17408, 5120), (synth.Q3_K, 17408, 5120),
]


@pytest.mark.parametrize("fmt,N,K", FULL, ids=[f"{synth.FORMAT_NAMES[f]}-{n}x{k}" for f, n, k in FULL])
def test_gemv_full_size_sampled(qg, fmt, N, K):
    g = np.random.default_rng(3000 + N + fmt)
    W = synth.weights(fmt, N, K, g)
    for M in (1, 4):
        x = synth.activations(M, K, g)
        y = host(qg.qg_gemv(fmt, dev(W), dev(x), N))
        rows = np.unique(np.concatenate([g.choice(N, size=min(N, 384), replace=False), [0, N - 1]]))
        Ws = W[rows]
        oq, od, os_ = oracle.quantize_act(x)
        y_ref = oracle.gemv_q(fmt, Ws, oq, od, os_, len(rows), K)
        sabs = oracle.absdot(fmt, Ws, oq, od, len(rows), K)
        assert_within(y[:, rows], y_ref, sabs, f"{synth.FORMAT_NAMES[fmt]} {N}x{K} M={M}")


# ----------------------------------------------------------------------------- properties
def test_gemv_deterministic_and_guard_bands(qg):
    import torch
    fmt, N, K, M = synth.Q4_K, 5120, 17408, 2
    g = np.random.default_rng(9)
    W = dev(synth.weights(fmt, N, K, g))
    x = dev(synth.activations(M, K, g))
    big = torch.full((M * N + 128,), float("nan"), device="cuda")
    y1 = big[64:64 + M * N].view(M, N)
    qg.qg_gemv(fmt, W, x, N, y=y1)
    y2 = qg.qg_gemv(fmt, W, x, N)
    torch.cuda.synchronize()
    assert torch.isnan(big[:64]).all() and torch.isnan(big[64 + M * N:]).all()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_power_of_two_scaling_exact(qg):
    fmt, N, K = synth.IQ4_XS, 2048, 4096
    g = np.random.default_rng(10)
    W = dev(synth.weights(fmt, N, K, g))
    x = synth.activations(1, K, g)
    y1 = host(qg.qg_gemv(fmt, W, dev(x), N))
    y8 = host(qg.qg_gemv(fmt, W, dev(x * np.float32(8)), N))
    np.testing.assert_array_equal(y8, y1 * 8)


def test_no_device_error_recorded(qg):
    assert qg.qg_device_error() == 0
