"""Pins of the CPU oracle to facts that do not come from the oracle itself.

* fp16 decoding against numpy's IEEE binary16 conversion (a library routine);
* hand-built blocks whose values were worked out by hand (tests/golden/blocks.txt);
* round trips through an encoder written here, independently of the decoder;
* the activation quantizer's rounding on hand-made exact ties;
* the integer-sum path against brute-force fp64 dequantize-then-dot (numpy matmul);
* exact scaling by powers of two (linearity where quantization keeps the codes);
* closed forms (all-ones Q8_0 weights reduce the GEMV to a plain sum);
* the router's top-k against a full stable sort, softmax invariants;
* SwiGLU identities (silu(g) - silu(-g) = g, silu(ln 3) = 0.75 ln 3);
* MoE special cases that reduce to the FFN sublayer;
* s16 activations: an exact grid (step 2^-20) with its ties, the step equal to the int8
  step / 256 bit for bit, the integer path against fp64 brute force, and an end-to-end
  MoE much closer than the int8 one to the unquantized fp64 MoE.
"""
import math
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "blocks.txt")
FMTS = [synth.Q4_0, synth.Q4_1, synth.Q5_0, synth.Q5_1, synth.Q8_0, synth.Q2_K, synth.Q3_K, synth.Q4_K,
        synth.Q5_K, synth.Q6_K, synth.IQ4_NL, synth.IQ4_XS]
MIN_FMTS = (synth.Q4_K, synth.Q5_K, synth.Q4_1, synth.Q5_1, synth.Q2_K)  # formats with a min term
IQ4NL = [-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113]


# ----------------------------------------------------------------------------- fp16
def test_half_to_double_matches_numpy(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ----------------------------------------------------------------------------- golden
def _parse_golden():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "block":
                cur = {"fmt": synth.FORMATS[tok[1]], "blk": np.zeros(int(tok[2]), np.uint8), "w": []}
            elif tok[0] == "byte":
                cur["blk"][int(tok[1])] = int(tok[2], 0)
            elif tok[0] == "w":
                cur["w"].append((int(tok[1]), float(tok[2])))
            elif tok[0] == "end":
                cases.append(cur)
                cur = None
    return cases


def test_golden_blocks(orc):
    cases = _parse_golden()
    assert {c["fmt"] for c in cases} == set(FMTS)
    for c in cases:
        w, _, _, _ = orc.decode_block(c["fmt"], c["blk"])
        for e, v in c["w"]:
            assert w[e] == v, (synth.FORMAT_NAMES[c["fmt"]], e, w[e], v)


# ----------------------------------------------------------------------------- encoders
def _h(v):
    return np.array([v], np.float16).view(np.uint8)


def _enc_q8_0(d, q):
    b = np.zeros(34, np.uint8)
    b[0:2] = _h(d)
    b[2:34] = np.asarray(q, np.int8).view(np.uint8)
    return b


def _enc_q4_0(d, nib):
    b = np.zeros(18, np.uint8)
    b[0:2] = _h(d)
    for i in range(16):
        b[2 + i] = nib[i] | (nib[16 + i] << 4)
    return b


def _enc_q4_1(d, m, nib):
    b = np.zeros(20, np.uint8)
    b[0:2] = _h(d)
    b[2:4] = _h(m)
    for i in range(16):
        b[4 + i] = nib[i] | (nib[16 + i] << 4)
    return b


def _enc_q5(fmt, d, m, code):
    """code[32] in 0..31 (stored): Q5_0 without m, Q5_1 with m."""
    one = fmt == synth.Q5_1
    b = np.zeros(24 if one else 22, np.uint8)
    b[0:2] = _h(d)
    if one:
        b[2:4] = _h(m)
    qh = sum(((int(code[e]) >> 4) & 1) << e for e in range(32))
    qo = 4 if one else 2
    b[qo:qo + 4] = np.array([qh & 255, (qh >> 8) & 255, (qh >> 16) & 255, qh >> 24], np.uint8)
    so = qo + 4
    for i in range(16):
        b[so + i] = (code[i] & 15) | ((code[16 + i] & 15) << 4)
    return b


def _enc_iq4_nl(d, idx):
    b = np.zeros(18, np.uint8)
    b[0:2] = _h(d)
    for i in range(16):
        b[2 + i] = idx[i] | (idx[16 + i] << 4)
    return b


def _pack_sc12(S, M):
    sc = np.zeros(12, np.uint8)
    for j in range(4):
        sc[j] = (S[j] & 63) | ((S[j + 4] >> 4) << 6)
        sc[j + 4] = (M[j] & 63) | ((M[j + 4] >> 4) << 6)
        sc[j + 8] = (S[j + 4] & 15) | ((M[j + 4] & 15) << 4)
    return sc


def _enc_q45_k(fmt, d, dmin, S, M, code):
    """code[256] in 0..15 (Q4_K) or 0..31 (Q5_K), element order."""
    b = np.zeros(synth.BLOCK_BYTES[fmt], np.uint8)
    b[0:2] = _h(d)
    b[2:4] = _h(dmin)
    b[4:16] = _pack_sc12(S, M)
    qs_off = 16 if fmt == synth.Q4_K else 48
    for e in range(256):
        j, l = divmod(e, 32)
        lo = code[e] & 15
        pos = qs_off + 32 * (j // 2) + l
        b[pos] |= lo if j % 2 == 0 else lo << 4
        if fmt == synth.Q5_K and code[e] >= 16:
            b[16 + l] |= 1 << j
    return b


def _enc_q6_k(d, sc, code):
    """code[256] in 0..63 (stored), sc[16] int8."""
    b = np.zeros(210, np.uint8)
    for e in range(256):
        h, r = divmod(e, 128)
        t, l = divmod(r, 32)
        lo, hi = code[e] & 15, code[e] >> 4
        pos = 64 * h + l + 32 * (t & 1)
        b[pos] |= lo if t < 2 else lo << 4
        b[128 + 32 * h + l] |= hi << (2 * t)
    b[192:208] = np.asarray(sc, np.int8).view(np.uint8)
    b[208:210] = _h(d)
    return b


def _enc_q2_k(d, dmin, S, M, code):
    """S[16], M[16] in 0..15 (per 16-element sub-block), code[256] in 0..3."""
    b = np.zeros(84, np.uint8)
    for s in range(16):
        b[s] = S[s] | (M[s] << 4)
    for e in range(256):
        h, r = divmod(e, 128)
        j, l = divmod(r, 32)
        b[16 + 32 * h + l] |= code[e] << (2 * j)
    b[80:82] = _h(d)
    b[82:84] = _h(dmin)
    return b


def _enc_q3_k(d, sc, q3):
    """sc[16] in -32..31 (per 16-element sub-block), q3[256] in -4..3."""
    b = np.zeros(110, np.uint8)
    for i in range(16):
        v = int(sc[i]) + 32
        if i < 8:
            b[96 + i] |= v & 15
        else:
            b[96 + i - 8] |= (v & 15) << 4
        b[104 + i % 4] |= (v >> 4) << (2 * (i // 4))
    for e in range(256):
        h, r = divmod(e, 128)
        j, l = divmod(r, 32)
        q = int(q3[e])
        b[32 + 32 * h + l] |= (q & 3) << (2 * j)
        if q >= 0:
            b[l] |= 1 << (4 * h + j)
    b[108:110] = _h(d)
    return b


def _enc_iq4_xs(d, ls, idx):
    b = np.zeros(136, np.uint8)
    b[0:2] = _h(d)
    sh = 0
    for ib in range(8):
        sh |= (ls[ib] >> 4) << (2 * ib)
        b[4 + ib // 2] |= (ls[ib] & 15) << (4 * (ib % 2))
    b[2] = sh & 255
    b[3] = sh >> 8
    for e in range(256):
        ib, j = divmod(e, 32)
        pos = 8 + 16 * ib + (j % 16)
        b[pos] |= idx[e] if j < 16 else idx[e] << 4
    return b


@pytest.mark.parametrize("fmt", FMTS)
def test_roundtrip_encode_decode(orc, fmt):
    g = np.random.default_rng(1234 + fmt)
    for _ in range(20):
        d = float(np.float16(g.uniform(0.25, 2.0)))
        if fmt == synth.Q8_0:
            q = g.integers(-127, 128, 32)
            blk, expect = _enc_q8_0(d, q), d * q
        elif fmt == synth.Q4_0:
            nib = g.integers(0, 16, 32)
            blk, expect = _enc_q4_0(d, nib), d * (nib - 8)
        elif fmt == synth.Q4_1:
            m = float(np.float16(g.uniform(-1, 1)))
            nib = g.integers(0, 16, 32)
            blk, expect = _enc_q4_1(d, m, nib), d * nib + m
        elif fmt in (synth.Q5_0, synth.Q5_1):
            m = float(np.float16(g.uniform(-1, 1)))
            code = g.integers(0, 32, 32)
            blk = _enc_q5(fmt, d, m, code)
            expect = d * (code - 16) if fmt == synth.Q5_0 else d * code + m
        elif fmt == synth.IQ4_NL:
            idx = g.integers(0, 16, 32)
            blk, expect = _enc_iq4_nl(d, idx), d * np.array(IQ4NL)[idx]
        elif fmt in (synth.Q4_K, synth.Q5_K):
            dmin = float(np.float16(g.uniform(0, 1)))
            S, M = g.integers(0, 64, 8), g.integers(0, 64, 8)
            code = g.integers(0, 16 if fmt == synth.Q4_K else 32, 256)
            blk = _enc_q45_k(fmt, d, dmin, S, M, code)
            j = np.arange(256) // 32
            expect = d * S[j] * code - dmin * M[j]
        elif fmt == synth.Q6_K:
            sc = g.integers(-127, 128, 16)
            code = g.integers(0, 64, 256)
            blk = _enc_q6_k(d, sc, code)
            expect = d * sc[np.arange(256) // 16] * (code - 32)
        elif fmt == synth.Q2_K:
            dmin = float(np.float16(g.uniform(0, 1)))
            S, M = g.integers(0, 16, 16), g.integers(0, 16, 16)
            code = g.integers(0, 4, 256)
            blk = _enc_q2_k(d, dmin, S, M, code)
            s = np.arange(256) // 16
            expect = d * S[s] * code - dmin * M[s]
        elif fmt == synth.Q3_K:
            sc = g.integers(-32, 32, 16)
            q3 = g.integers(-4, 4, 256)
            blk = _enc_q3_k(d, sc, q3)
            expect = d * sc[np.arange(256) // 16] * q3
        else:
            ls = g.integers(0, 64, 8)
            idx = g.integers(0, 16, 256)
            blk = _enc_iq4_xs(d, ls, idx)
            expect = d * (ls[np.arange(256) // 32] - 32) * np.array(IQ4NL)[idx]
        w, c, A, B, mc = orc.decode_block(fmt, blk, with_mc=True)
        np.testing.assert_array_equal(w, expect)
        # the integer decomposition rebuilds the same weights
        u = np.arange(len(w)) // 32
        np.testing.assert_allclose(A[u] * c - B[u] * mc, w, rtol=0, atol=1e-12 * (1 + np.abs(w).max()))


def test_q3k_each_scale_alone(orc):
    """Each of the 16 packed 6-bit scales (both nibble paths, all four high-bit pairs)
    selects exactly its own 16 elements."""
    for i in range(16):
        for v in (-32, -31, -17, 1, 15, 31):
            sc = [0] * 16
            sc[i] = v
            w, _, _, _ = orc.decode_block(synth.Q3_K, _enc_q3_k(1.0, sc, [3] * 256))
            nz = np.flatnonzero(w)
            if v:
                np.testing.assert_array_equal(nz, np.arange(16 * i, 16 * i + 16))
                assert np.all(w[nz] == 3 * v)
            else:
                assert nz.size == 0


def test_q2k_scale_and_min_nibbles(orc):
    """Q2_K: the low nibble scales the code, the high nibble is the min, per 16 elements."""
    for s in range(16):
        S, M = [0] * 16, [0] * 16
        S[s], M[s] = 5, 3
        w, _, _, _ = orc.decode_block(synth.Q2_K, _enc_q2_k(1.0, 1.0, S, M, [2] * 256))
        nz = np.flatnonzero(w)
        np.testing.assert_array_equal(nz, np.arange(16 * s, 16 * s + 16))
        assert np.all(w[nz] == 5 * 2 - 3)


def test_iq4_codebook_recovered(orc):
    idx = np.array([i % 16 for i in range(256)])
    blk = _enc_iq4_xs(1.0, [33] * 8, idx)     # scale d*(33-32) = 1
    w, c, _, _ = orc.decode_block(synth.IQ4_XS, blk)
    np.testing.assert_array_equal(w[:16], IQ4NL)
    np.testing.assert_array_equal(c[:16], IQ4NL)


def test_single_nonzero_subblock_kquant(orc):
    """Each of the 8 sub-blocks (both 6-bit packing paths) selected alone."""
    for fmt in (synth.Q4_K, synth.Q5_K):
        for j in range(8):
            for s in (1, 17, 33, 63):
                S = [0] * 8
                S[j] = s
                blk = _enc_q45_k(fmt, 1.0, 0.0, S, [0] * 8, [15] * 256)
                w, _, _, _ = orc.decode_block(fmt, blk)
                nz = np.flatnonzero(w)
                np.testing.assert_array_equal(nz, np.arange(32 * j, 32 * j + 32))
                assert np.all(w[nz] == 15 * s)


# ----------------------------------------------------------------------------- activation quant
def test_quant_zero_block(orc):
    xq, xd, xs = orc.quantize_act(np.zeros((1, 64), np.float32))
    assert not xq.any() and not xd.any() and not xs.any()


def test_quant_single_nonzero(orc):
    for a in (3.0, -3.0, 1e-20, 7.5e5):
        x = np.zeros((1, 32), np.float32)
        x[0, 5] = a
        xq, xd, xs = orc.quantize_act(x)
        assert xq[0, 5] == (127 if a > 0 else -127)
        assert np.count_nonzero(xq) == 1
        assert xd[0, 0] == np.float32(abs(np.float32(a))) / np.float32(127)
        assert xs[0, 0] == xq[0, 5]


def test_quant_half_ties_round_away_from_zero(orc):
    # amax = 127 makes d = 1 exactly, so q = round(x) with exact ties
    vals = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 3.4999998, 0.49999997, 126.5]
    want = [127, 3, -3, 1, -1, 2, -2, 3, 0, 127]
    x = np.zeros((1, 32), np.float32)
    x[0, :len(vals)] = vals
    xq, xd, xs = orc.quantize_act(x)
    assert xd[0, 0] == 1.0
    assert list(xq[0, :len(vals)]) == want
    assert xs[0, 0] == sum(want)


def _half_away(v):
    v = v.astype(np.float64)                      # exact for fp32 values
    return (np.sign(v) * np.floor(np.abs(v) + 0.5)).astype(np.int64)


def test_quant_uses_true_division(orc):
    """Blocks where fp32 x/d and x*(1/d) round to different codes: the codes must be
    the ones of the IEEE division (numpy's fp32 division is correctly rounded)."""
    g = np.random.default_rng(2024)
    amax = g.uniform(0.5, 4.0, size=64).astype(np.float32)
    d = (amax / np.float32(127)).astype(np.float32)
    k = np.arange(126)
    blocks = []
    for i in range(len(amax)):
        near = ((k + 0.5) * np.float64(d[i])).astype(np.float32)      # values near code ties
        cand = np.concatenate([near, np.nextafter(near, np.float32(np.inf)),
                               np.nextafter(near, np.float32(-np.inf))])
        vd = (cand / d[i]).astype(np.float32)
        vr = (cand * (np.float32(1) / d[i])).astype(np.float32)
        diff = cand[_half_away(vd) != _half_away(vr)]
        if diff.size:
            blk = np.zeros(32, np.float32)
            blk[0] = amax[i]
            blk[1:1 + min(31, diff.size)] = diff[:31]
            blocks.append(blk)
    assert len(blocks) >= 8
    x = np.stack(blocks)
    dd = (np.abs(x).max(1) / np.float32(127)).astype(np.float32)[:, None]
    want = np.clip(_half_away((x / dd).astype(np.float32)), -127, 127)
    xq, xd, _ = orc.quantize_act(x.reshape(1, -1))
    np.testing.assert_array_equal(xq.reshape(-1, 32), want)
    np.testing.assert_array_equal(xd.reshape(-1), dd[:, 0])


def test_quant_properties(orc):
    g = np.random.default_rng(7)
    x = (g.standard_normal((5, 512)) * np.exp(g.uniform(-20, 20, (5, 1)))).astype(np.float32)
    xq, xd, xs = orc.quantize_act(x)
    xb = x.reshape(5, 16, 32).astype(np.float64)
    qb = xq.reshape(5, 16, 32).astype(np.int64)
    amax = np.abs(x.reshape(5, 16, 32)).max(-1)
    np.testing.assert_array_equal(xd, (amax / np.float32(127)).astype(np.float32))
    assert np.all(np.abs(qb).max(-1) == 127)
    assert np.all(np.abs(xb - qb * xd[..., None].astype(np.float64)) <= 0.5 * xd[..., None] * (1 + 1e-6))
    np.testing.assert_array_equal(xs, qb.sum(-1))


# ----------------------------------------------------------------------------- GEMV paths
@pytest.mark.parametrize("fmt", FMTS)
def test_int_path_equals_fp64_bruteforce(orc, fmt):
    g = np.random.default_rng(99 + fmt)
    qk = synth.BLOCK_ELEMS[fmt]
    for N, K, M in [(3, qk, 1), (5, 2 * qk, 2), (8, 512 if qk == 256 else 96, 3)]:
        W = synth.weights(fmt, N, K, g)
        x = synth.activations(M, K, g)
        xq, xd, xs = orc.quantize_act(x)
        y_int = orc.gemv_q(fmt, W, xq, xd, xs, N, K)
        y_deq = orc.gemv_deq(fmt, W, xq, xd, N, K)
        Wd = orc.dequant_matrix(fmt, W, N, K)
        xhat = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1)
        y_np = xhat @ Wd.T
        sabs = orc.absdot(fmt, W, xq, xd, N, K)
        np.testing.assert_allclose(sabs, np.abs(xhat)[:, None, :].__mul__(np.abs(Wd)[None]).sum(-1), rtol=1e-12)
        tol = 1e-12 * sabs + 1e-300
        assert np.all(np.abs(y_int - y_deq) <= tol)
        assert np.all(np.abs(y_int - y_np) <= tol)
        # block dots rebuild the same y
        dots, aux = orc.block_dots(fmt, W, xq, xs, N, K)
        codes = np.stack([np.concatenate([orc.decode_block(fmt, W[n, b * synth.BLOCK_BYTES[fmt]:(b + 1) * synth.BLOCK_BYTES[fmt]])[1]
                                          for b in range(K // qk)]) for n in range(N)])
        want = np.einsum("nuk,muk->mnu", codes.reshape(N, K // 32, 32).astype(np.int64),
                         xq.reshape(M, K // 32, 32).astype(np.int64))
        np.testing.assert_array_equal(dots, want)
        if fmt == synth.Q2_K:  # per-16 mins: aux is the unit's sum of min code * activation code
            mcs = np.stack([np.concatenate([orc.decode_block(fmt, W[n, b * 84:(b + 1) * 84], with_mc=True)[4]
                                            for b in range(K // qk)]) for n in range(N)])
            want_a = np.einsum("nuk,muk->mnu", mcs.reshape(N, K // 32, 32).astype(np.int64),
                               xq.reshape(M, K // 32, 32).astype(np.int64))
            np.testing.assert_array_equal(aux, want_a)
        elif fmt in MIN_FMTS:
            np.testing.assert_array_equal(aux, np.broadcast_to(xs[:, None, :], aux.shape))
        else:
            assert not aux.any()


@pytest.mark.parametrize("fmt", FMTS)
def test_power_of_two_scaling_is_exact(orc, fmt):
    g = np.random.default_rng(5 + fmt)
    N, K = 4, 512
    W = synth.weights(fmt, N, K, g)
    x = synth.activations(2, K, g)
    y1 = orc.gemv(fmt, W, x, N, K)
    for p in (-3, 1, 4):
        yp = orc.gemv(fmt, W, (x * np.float32(2.0 ** p)).astype(np.float32), N, K)
        np.testing.assert_array_equal(yp, y1 * 2.0 ** p)


def test_q8_all_ones_is_a_plain_sum(orc):
    N, K = 3, 128
    blk = _enc_q8_0(1.0, [1] * 32)
    W = np.tile(blk, (N, K // 32))
    g = np.random.default_rng(3)
    x = g.integers(-126, 127, size=(2, K)).astype(np.float32)
    x[:, ::32] = 127.0                   # amax 127 in every block: d = 1, q = x
    y = orc.gemv(synth.Q8_0, W, x, N, K)
    np.testing.assert_array_equal(y, np.repeat(x.sum(1, keepdims=True).astype(np.float64), N, axis=1))


# ----------------------------------------------------------------------------- router
def test_router_topk_matches_full_sort(orc):
    g = np.random.default_rng(11)
    E, H, k = 256, 2048, 8
    Wr = synth.router_weights(E, H, g)
    x = synth.activations(4, H, g)
    logits, p, ids, w = orc.router(x, Wr, k)
    for m in range(4):
        order = np.argsort(-p[m], kind="stable")
        np.testing.assert_array_equal(ids[m], order[:k])
        np.testing.assert_allclose(w[m], p[m, order[:k]] / p[m, order[:k]].sum(), rtol=1e-15)
        assert abs(p[m].sum() - 1) < 1e-13 and abs(w[m].sum() - 1) < 1e-13
        i, j = ids[m, 0], ids[m, 5]
        assert math.isclose(p[m, i] / p[m, j], math.exp(logits[m, i] - logits[m, j]), rel_tol=1e-12)
    ref_logits = x.astype(np.float64) @ Wr.astype(np.float64).T
    np.testing.assert_allclose(logits, ref_logits, rtol=1e-12, atol=1e-12)


def test_router_tie_prefers_lower_id(orc):
    E, H = 16, 32
    Wr = np.zeros((E, H), np.float32)
    for e in (3, 7, 9, 12):
        Wr[e, 0] = 1.0                     # four experts with identical logits
    Wr[5, 0] = 2.0
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    _, _, ids, w = orc.router(x, Wr, 3)
    assert list(ids[0]) == [5, 3, 7]


# ----------------------------------------------------------------------------- swiglu
def test_swiglu_identities(orc):
    assert orc.swiglu(0.0, 5.0) == 0.0
    for gv in (0.1, 1.0, 3.7, 25.0):
        assert math.isclose(orc.swiglu(gv, 1.0) - orc.swiglu(-gv, 1.0), gv, rel_tol=1e-14)
    assert math.isclose(orc.swiglu(math.log(3.0), 1.0), 0.75 * math.log(3.0), rel_tol=1e-15)
    assert math.isclose(orc.swiglu(1.3, 4.0), 4.0 * orc.swiglu(1.3, 1.0), rel_tol=1e-15)


def test_requant_is_quant_of_fp32(orc):
    g = np.random.default_rng(4)
    h = g.standard_normal((3, 64)) * 3
    a = orc.requant(h)
    b = orc.quantize_act(h.astype(np.float32))
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


# ----------------------------------------------------------------------------- MoE / FFN
def _moe_small(g, fmt, E, H, I):
    Wg = synth.stacked_experts(fmt, E, I, H, g)
    Wu = synth.stacked_experts(fmt, E, I, H, g)
    Wd = synth.stacked_experts(fmt, E, H, I, g)
    sh = (synth.weights(fmt, I, H, g), synth.weights(fmt, I, H, g), synth.weights(fmt, H, I, g))
    return Wg, Wu, Wd, sh


def test_moe_single_expert_reduces_to_two_ffns(orc):
    g = np.random.default_rng(21)
    fmt, E, H, I, M = synth.Q4_K, 1, 512, 256, 2
    Wg, Wu, Wd, (sg, su, sd) = _moe_small(g, fmt, E, H, I)
    Wr = synth.router_weights(E, H, g)
    x = synth.activations(M, H, g)
    y, ids, w = orc.moe_ffn(fmt, x, Wr, 1, Wg, Wu, Wd, sg, su, sd, I)
    assert np.all(ids == 0) and np.all(w == 1.0)
    ye = orc.ffn_sublayer(fmt, Wg[0], Wu[0], Wd[0], x, I)[0]
    ys = orc.ffn_sublayer(fmt, sg, su, sd, x, I)[0]
    np.testing.assert_array_equal(y, ye + ys)


def test_moe_identical_experts_ignore_router(orc):
    g = np.random.default_rng(22)
    fmt, E, H, I, M, k = synth.Q4_0, 6, 256, 64, 3, 2
    one = _moe_small(g, fmt, 1, H, I)
    Wg = np.repeat(one[0], E, axis=0)
    Wu = np.repeat(one[1], E, axis=0)
    Wd = np.repeat(one[2], E, axis=0)
    sg, su, sd = one[3]
    Wr = synth.router_weights(E, H, g)
    x = synth.activations(M, H, g)
    y, ids, w = orc.moe_ffn(fmt, x, Wr, k, Wg, Wu, Wd, sg, su, sd, I)
    ye = orc.ffn_sublayer(fmt, one[0][0], one[1][0], one[2][0], x, I)[0]
    ys = orc.ffn_sublayer(fmt, sg, su, sd, x, I)[0]
    np.testing.assert_allclose(y, ye + ys, rtol=1e-12, atol=1e-12 * np.abs(ye).max())


def test_moe_stages_compose(orc):
    g = np.random.default_rng(23)
    fmt, E, H, I, M, k = synth.Q4_K, 8, 512, 256, 2, 3
    Wg, Wu, Wd, (sg, su, sd) = _moe_small(g, fmt, E, H, I)
    Wr = synth.router_weights(E, H, g)
    x = synth.activations(M, H, g)
    y, ids, w = orc.moe_ffn(fmt, x, Wr, k, Wg, Wu, Wd, sg, su, sd, I)
    _, _, ids2, w2 = orc.router(x, Wr, k)
    gg, uu, hh = orc.moe_gateup(fmt, x, E, k, I, ids2, Wg, Wu, sg, su)
    hq, hd, hs = orc.requant(hh.reshape(M * (k + 1), I))
    y2, yabs = orc.moe_down(fmt, M, H, E, k, I, ids2, w2, hq, hd, hs, Wd, sd)
    np.testing.assert_array_equal(ids, ids2)
    np.testing.assert_array_equal(y, y2)
    # a routed slot's g equals the plain GEMV of that expert
    xq, xd, xs = orc.quantize_act(x)
    e = ids[1, 2]
    ref = orc.gemv_q(fmt, Wg[e], xq[1:2], xd[1:2], xs[1:2], I, H)[0]
    np.testing.assert_array_equal(gg[1, 2], ref)
    assert np.all(yabs >= np.abs(y) * (1 - 1e-12))


# ----------------------------------------------------------------------------- s16 activations
def test_quant16_exact_grid(orc):
    """amax = 32512 * 2^-20 makes the s16 step d = 2^-20 exactly: elements on the grid
    j * 2^-20 quantize to j, exact half steps round away from zero."""
    step = 2.0 ** -20
    j = [32512, -12345, 0, 1, -1, 255, 256, -257, 20000, -32511]
    ties = [2.5, -2.5, 0.5, -0.5, 32511.5, -100.5]
    want_t = [3, -3, 1, -1, 32512, -101]
    x = np.zeros((1, 32), np.float32)
    x[0, :len(j)] = np.array(j, np.float64) * step
    x[0, len(j):len(j) + len(ties)] = np.array(ties, np.float64) * step
    xq, xd, xs = orc.quantize_act16(x)
    assert xd[0, 0] == np.float32(step)
    want = j + want_t + [0] * (32 - len(j) - len(ties))
    assert list(xq[0]) == want
    assert xs[0, 0] == sum(want)


def test_quant16_step_is_int8_step_over_256(orc):
    """The s16 step is the int8 step divided by 256, bit for bit."""
    g = np.random.default_rng(8)
    x = (g.standard_normal((4, 1024)) * np.exp(g.uniform(-20, 20, (4, 1)))).astype(np.float32)
    _, d8, _ = orc.quantize_act(x)
    _, d16, _ = orc.quantize_act16(x)
    np.testing.assert_array_equal(d16, (d8 / np.float32(256)).astype(np.float32))


def test_quant16_properties(orc):
    g = np.random.default_rng(9)
    x = (g.standard_normal((5, 512)) * np.exp(g.uniform(-20, 20, (5, 1)))).astype(np.float32)
    x[1, 32:64] = 0.0
    xq, xd, xs = orc.quantize_act16(x)
    xb = x.reshape(5, 16, 32).astype(np.float64)
    qb = xq.reshape(5, 16, 32).astype(np.int64)
    amax = np.abs(x.reshape(5, 16, 32)).max(-1)
    np.testing.assert_array_equal(xd, (amax / np.float32(32512)).astype(np.float32))
    nz = amax > 0
    assert np.all(np.abs(qb).max(-1)[nz] == 32512) and not qb[~nz].any()
    # x/d is rounded to fp32 before the code is taken: up to 32512 * 2^-24 of a step off
    bound = (0.5 + 32512 * 2.0 ** -23) * xd[..., None].astype(np.float64)
    assert np.all(np.abs(xb - qb * xd[..., None].astype(np.float64)) <= bound)
    np.testing.assert_array_equal(xs, qb.sum(-1))


def test_requant16_is_quant16_of_fp32(orc):
    g = np.random.default_rng(10)
    h = g.standard_normal((3, 64)) * 3
    for u, v in zip(orc.requant16(h), orc.quantize_act16(h.astype(np.float32))):
        np.testing.assert_array_equal(u, v)


@pytest.mark.parametrize("fmt", FMTS)
def test_int16_path_equals_fp64_bruteforce(orc, fmt):
    """s16 codes through the integer-sum path equal fp64 dequantize-then-dot, and the
    s16 result is far closer to the unquantized product than the int8 one."""
    g = np.random.default_rng(199 + fmt)
    qk = synth.BLOCK_ELEMS[fmt]
    N, K, M = 6, 512 if qk == 256 else 128, 2
    W = synth.weights(fmt, N, K, g)
    x = synth.activations(M, K, g)
    xq, xd, xs = orc.quantize_act16(x)
    Wd = orc.dequant_matrix(fmt, W, N, K)
    xhat = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1)
    y16 = orc.gemv_q16(fmt, W, xq, xd, xs, N, K)
    sabs = orc.absdot16(fmt, W, xq, xd, N, K)
    np.testing.assert_allclose(sabs, (np.abs(xhat)[:, None, :] * np.abs(Wd)[None]).sum(-1), rtol=1e-12)
    assert np.all(np.abs(y16 - xhat @ Wd.T) <= 1e-12 * sabs + 1e-300)
    y_exact = x.astype(np.float64) @ Wd.T
    y8 = orc.gemv(fmt, W, x, N, K)
    assert np.abs(y16 - y_exact).max() * 50 < np.abs(y8 - y_exact).max()


def _moe_exact(orc, fmt, x, Wr, k, Wg, Wu, Wd, sg, su, sd, I):
    """fp64 MoE FFN with unquantized activations, from the dequantized matrices."""
    M, H = x.shape
    _, _, ids, w = orc.router(x, Wr, k)
    deq = lambda W, n, kk: orc.dequant_matrix(fmt, W, n, kk)  # noqa: E731
    y = np.zeros((M, H))
    for m in range(M):
        xm = x[m].astype(np.float64)
        for s in range(k + 1):
            Wg_s, Wu_s, Wd_s = (Wg[ids[m, s]], Wu[ids[m, s]], Wd[ids[m, s]]) if s < k else (sg, su, sd)
            gg, uu = deq(Wg_s, I, H) @ xm, deq(Wu_s, I, H) @ xm
            h = gg * uu / (1 + np.exp(-gg))
            y[m] += (w[m, s] if s < k else 1.0) * (deq(Wd_s, H, I) @ h)
    return y


def test_moe16_stages_compose_and_beat_int8(orc):
    g = np.random.default_rng(24)
    fmt, E, H, I, M, k = synth.Q4_K, 8, 512, 256, 2, 3
    Wg, Wu, Wd, (sg, su, sd) = _moe_small(g, fmt, E, H, I)
    Wr = synth.router_weights(E, H, g)
    x = synth.activations(M, H, g)
    y, ids, w = orc.moe_ffn16(fmt, x, Wr, k, Wg, Wu, Wd, sg, su, sd, I)
    _, _, ids2, w2 = orc.router(x, Wr, k)
    gg, uu, hh = orc.moe_gateup16(fmt, x, E, k, I, ids2, Wg, Wu, sg, su)
    hq, hd, hs = orc.requant16(hh.reshape(M * (k + 1), I))
    y2, yabs = orc.moe_down16(fmt, M, H, E, k, I, ids2, w2, hq, hd, hs, Wd, sd)
    np.testing.assert_array_equal(ids, ids2)
    np.testing.assert_array_equal(y, y2)
    xq, xd, xs = orc.quantize_act16(x)
    e = ids[1, 2]
    np.testing.assert_array_equal(gg[1, 2], orc.gemv_q16(fmt, Wg[e], xq[1:2], xd[1:2], xs[1:2], I, H)[0])
    np.testing.assert_array_equal(uu[0, k], orc.gemv_q16(fmt, su, xq[0:1], xd[0:1], xs[0:1], I, H)[0])
    assert np.all(yabs >= np.abs(y) * (1 - 1e-12))
    # the finer step shows end to end: the s16 MoE is much closer to the unquantized one
    y_exact = _moe_exact(orc, fmt, x, Wr, k, Wg, Wu, Wd, sg, su, sd, I)
    y8 = orc.moe_ffn(fmt, x, Wr, k, Wg, Wu, Wd, sg, su, sd, I)[0]
    assert np.abs(y - y_exact).max() * 50 < np.abs(y8 - y_exact).max()


# ----------------------------------------------------------------------------- prefill, fp16 operands
def _f16_probe_values():
    """fp32 inputs for the fp32 -> fp16 rounding: every finite fp16 value, every midpoint
    between neighbouring finite fp16 values (exact ties in fp32), the fp32 neighbours of
    those midpoints, the overflow boundary and values spread over 60 binades."""
    h = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)  # +0 .. 65504
    mids = (h[:-1] + h[1:]) / 2
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)                            # exact ties
    up = np.nextafter(mids32, np.float32(np.inf))
    down = np.nextafter(mids32, np.float32(0))
    edge = np.array([65504, 65519.99, 65520, 65536, 1e6, 2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -26,
                     2.0 ** -14, 2.0 ** -14 - 2.0 ** -25], np.float32)
    g = np.random.default_rng(1616)
    spread = (g.standard_normal(20000) * 2.0 ** g.integers(-40, 18, 20000)).astype(np.float32)
    v = np.concatenate([h.astype(np.float32), mids32, up, down, edge, spread])
    return np.concatenate([v, -v])


def test_float_to_half_matches_numpy(orc):
    x = _f16_probe_values()
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = orc.float_to_half(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[0]]!r}: {got[bad[0]]:#06x} vs {ref[bad[0]]:#06x}"


@pytest.mark.parametrize("fmt", FMTS)
def test_dequant_f16_is_rounded_fp32_weight(orc, fmt):
    # every product A*c and B*mc is exact in fp32 and their fp64 difference is exact, so
    # the reading's fp16 weight is numpy's fp64 -> fp32 -> fp16 rounding of the fp64 weight
    qk = synth.BLOCK_ELEMS[fmt]
    N, K = 7, 4 * qk
    W = synth.weights(fmt, N, K, np.random.default_rng(900 + fmt))
    w64 = orc.dequant_matrix(fmt, W, N, K)
    ref = w64.astype(np.float32).astype(np.float16).view(np.uint16)
    got = orc.dequant_f16(fmt, W, N, K)
    np.testing.assert_array_equal(got, ref)
    if fmt not in MIN_FMTS:  # one product only: w64 is exact in fp32, the fp16 rounding is direct
        np.testing.assert_array_equal(got, w64.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("fmt", FMTS)
def test_prefill_gemm_equals_fp64_matmul(orc, fmt):
    qk = synth.BLOCK_ELEMS[fmt]
    N, K, M = 9, 2 * max(qk, 128), 5
    g = np.random.default_rng(300 + fmt)
    W = synth.weights(fmt, N, K, g)
    x = synth.activations(M, K, g) * np.float32(3.0)
    w16 = orc.dequant_f16(fmt, W, N, K).view(np.float16).astype(np.float64)
    x16 = x.astype(np.float16).astype(np.float64)
    y, sabs = orc.prefill_gemm(fmt, W, x, N, K)
    np.testing.assert_allclose(y, x16 @ w16.T, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(sabs, np.abs(x16) @ np.abs(w16).T, rtol=1e-12, atol=1e-300)


def test_prefill_q8_integer_closed_form(orc):
    # Q8_0 with d = 1 (fp16 0x3c00): the fp16 weights are the int8 codes themselves, and
    # integer activations below 2048 are exact in fp16, so y is the integer dot product
    K, N, M = 64, 3, 2
    g = np.random.default_rng(5)
    codes = g.integers(-127, 128, (N, K)).astype(np.int8)
    W = np.zeros((N, K // 32, 34), np.uint8)
    W[:, :, 0], W[:, :, 1] = 0x00, 0x3c
    W[:, :, 2:] = codes.reshape(N, K // 32, 32).view(np.uint8)
    x = g.integers(-2047, 2048, (M, K)).astype(np.float32)
    y, _ = orc.prefill_gemm(synth.Q8_0, W.reshape(N, -1), x, N, K)
    want = x.astype(np.int64) @ codes.astype(np.int64).T
    np.testing.assert_array_equal(y, want.astype(np.float64))
