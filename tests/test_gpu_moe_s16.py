"""GPU parity of the MoE FFN with s16 activations (qg_moe_ffn_s16) and of the s16 activation
quantizer (qg_quantize_act_s16) against the CPU oracle.

  quantizer  codes, steps and code sums equal the oracle's s16 rule bit for bit;
  router     as for the int8 MoE (fp32 logits from fp32 x);
  gate/up    g and u, the fp32 sum of the two planes' partial rows, within
             1e-5 * sum|w*xhat| + 1e-6 of the oracle's s16 integer path (GPU's ids);
  swiglu     h within fp32 rounding of silu(g)*u evaluated in fp64 on the GPU's g, u;
  requant    the GPU's int16 codes equal the oracle's s16 quantization of the GPU's h;
  down       y within 1e-5 * sum|w|*sum|wd*hhat| + 1e-6 of the oracle on the GPU's codes;
  precision  end to end, the s16 result is much closer than the int8 one to the fp64 MoE
             with unquantized activations (the reason for the s16 variant).
"""
import numpy as np
import pytest

import oracle
import synth
from qg_testlib import FMT_IDS, FMTS, assert_within, dev, host, qg_module
from test_gpu_moe_ffn import _check_router, _ws_view

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    return qg_module()


def test_quantize_act_s16_bit_exact(qg):
    g = np.random.default_rng(1601)
    x = (g.standard_normal((7, 1024)) * np.exp(g.uniform(-25, 25, (7, 1)))).astype(np.float32)
    x[2, 64:96] = 0.0                                   # an all-zero block
    x[3, :32] = np.arange(-16, 16, dtype=np.float32) * np.float32(2.0 ** -20)  # exact grid
    xq, xd, xs = qg.qg_quantize_act_s16(dev(x))
    rq, rd, rs = oracle.quantize_act16(x)
    np.testing.assert_array_equal(host(xq), rq)
    np.testing.assert_array_equal(host(xd).view(np.uint32), rd.view(np.uint32))
    np.testing.assert_array_equal(host(xs), rs)


def _moe16_case(qg, fmt, M, H, E, topk, I, seed):
    import torch
    g = np.random.default_rng(seed)
    inp = dict(Wg=synth.stacked_experts(fmt, E, I, H, g), Wu=synth.stacked_experts(fmt, E, I, H, g),
               Wd=synth.stacked_experts(fmt, E, H, I, g))
    inp.update(sg=synth.weights(fmt, I, H, g), su=synth.weights(fmt, I, H, g), sd=synth.weights(fmt, H, I, g))
    inp.update(Wr=synth.router_weights(E, H, g), x=synth.activations(M, H, g))
    W = {k: dev(v) for k, v in inp.items()}
    nws = qg.qg_workspace_size(qg.QG_OP_MOE_FFN_S16, fmt, M, H, H, E, topk, I)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    ids = torch.empty((M, topk), dtype=torch.int32, device="cuda")
    w = torch.empty((M, topk), dtype=torch.float32, device="cuda")
    y = qg.qg_moe_ffn_s16(fmt, W["x"], W["Wr"], topk, W["Wg"], W["Wu"], W["Wd"], W["sg"], W["su"], W["sd"], I,
                          topk_ids=ids, topk_w=w, ws=ws)
    torch.cuda.synchronize()
    S = topk + 1
    off = qg.qg_moe_s16_ws_layout(M, H, E, topk, I)
    gp = _ws_view(ws, off[0], M * S * 2 * I, np.float32).reshape(M, S, 2, I)
    up = _ws_view(ws, off[1], M * S * 2 * I, np.float32).reshape(M, S, 2, I)
    out = dict(
        y=host(y), ids=host(ids), w=host(w),
        g=(gp[:, :, 0] + gp[:, :, 1]).astype(np.float32),        # fp32 adds, as on the GPU
        u=(up[:, :, 0] + up[:, :, 1]).astype(np.float32),
        h=_ws_view(ws, off[2], M * S * I, np.float32).reshape(M, S, I),
        hq=_ws_view(ws, off[3], M * S * I, np.int16).reshape(M * S, I),
        hd=_ws_view(ws, off[4], M * S * I // 32, np.float32).reshape(M * S, I // 32),
        hs=_ws_view(ws, off[5], M * S * I // 32, np.int32).reshape(M * S, I // 32),
        logits=_ws_view(ws, off[6], M * E, np.float32).reshape(M, E))
    return inp, out


def _moe_exact(inp, fmt, ids, w, topk, I):
    """fp64 MoE with unquantized activations, from the dequantized matrices and the ids and
    weights given."""
    x = inp["x"].astype(np.float64)
    M, H = x.shape
    y = np.zeros((M, H))
    for m in range(M):
        for s in range(topk + 1):
            Wg, Wu, Wd = ((inp["Wg"][ids[m, s]], inp["Wu"][ids[m, s]], inp["Wd"][ids[m, s]]) if s < topk
                          else (inp["sg"], inp["su"], inp["sd"]))
            gg = oracle.dequant_matrix(fmt, Wg, I, H) @ x[m]
            uu = oracle.dequant_matrix(fmt, Wu, I, H) @ x[m]
            h = gg * uu / (1 + np.exp(-gg))
            y[m] += (w[m, s] if s < topk else 1.0) * (oracle.dequant_matrix(fmt, Wd, H, I) @ h)
    return y


def _check_moe16(fmt, inp, out, M, H, E, topk, I):
    S = topk + 1
    x = inp["x"]
    _check_router(x, inp["Wr"], out, topk)
    ids = out["ids"].astype(np.int32)
    g_ref, u_ref, _ = oracle.moe_gateup16(fmt, x, E, topk, I, ids, inp["Wg"], inp["Wu"], inp["sg"], inp["su"])
    xq, xd, _ = oracle.quantize_act16(x)
    for m in range(M):
        for s in range(S):
            e = ids[m, s] if s < topk else None
            Wg_e = inp["Wg"][e] if e is not None else inp["sg"]
            Wu_e = inp["Wu"][e] if e is not None else inp["su"]
            ag = oracle.absdot16(fmt, Wg_e, xq[m:m + 1], xd[m:m + 1], I, H)[0]
            au = oracle.absdot16(fmt, Wu_e, xq[m:m + 1], xd[m:m + 1], I, H)[0]
            assert_within(out["g"][m, s], g_ref[m, s], ag, f"g m={m} s={s}")
            assert_within(out["u"][m, s], u_ref[m, s], au, f"u m={m} s={s}")
    gg, uu = out["g"].astype(np.float64), out["u"].astype(np.float64)
    h_exact = gg * uu / (1 + np.exp(-gg))
    assert np.all(np.abs(out["h"] - h_exact) <= 1e-6 * np.abs(h_exact) + 1e-30)
    hq, hd, hs = oracle.requant16(out["h"].reshape(M * S, I).astype(np.float64))
    np.testing.assert_array_equal(out["hq"], hq)
    np.testing.assert_array_equal(out["hd"].view(np.uint32), hd.view(np.uint32))
    np.testing.assert_array_equal(out["hs"], hs)
    y_ref, yabs = oracle.moe_down16(fmt, M, H, E, topk, I, ids, out["w"].astype(np.float64), out["hq"], out["hd"],
                                    out["hs"], inp["Wd"], inp["sd"])
    r = assert_within(out["y"], y_ref, yabs, "moe s16 y")
    y_pure, _, _ = oracle.moe_ffn16(fmt, x, inp["Wr"], topk, inp["Wg"], inp["Wu"], inp["Wd"], inp["sg"], inp["su"],
                                    inp["sd"], I)
    rel = np.abs(out["y"] - y_pure).max() / (np.abs(y_pure).max() + 1e-30)
    print(f"moe s16 fmt={fmt} M={M}: worst err/bound {r:.3f}, end-to-end max rel {rel:.2e}")


@pytest.mark.parametrize("M", [1, 2, 4])
def test_moe_s16_config_shape(qg, M):
    """256 routed experts + 1 shared, hidden 2048, inter 512, top-8, Q4_K."""
    fmt, H, E, topk, I = synth.Q4_K, 2048, 256, 8, 512
    inp, out = _moe16_case(qg, fmt, M, H, E, topk, I, seed=synth.seed_for(4, 16 + M))
    _check_moe16(fmt, inp, out, M, H, E, topk, I)


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_moe_s16_formats_small(qg, fmt):
    M, H, E, topk, I = 3, 512, 40, 4, 256
    inp, out = _moe16_case(qg, fmt, M, H, E, topk, I, seed=1600 + fmt)
    _check_moe16(fmt, inp, out, M, H, E, topk, I)


def test_moe_s16_large_batch_chunks(qg):
    """16 tokens x 9 slots x 2 planes of h exceed one CTA's shared memory: the down
    projection runs in token chunks."""
    fmt, M, H, E, topk, I = synth.Q4_K, 16, 2048, 64, 8, 1024
    inp, out = _moe16_case(qg, fmt, M, H, E, topk, I, seed=1677)
    _check_moe16(fmt, inp, out, M, H, E, topk, I)


def test_moe_s16_is_closer_to_unquantized(qg):
    """On the same routing, the s16 MoE lands much closer than the int8 one to the fp64 MoE
    whose activations are not quantized at all."""
    import torch
    fmt, M, H, E, topk, I = synth.Q4_K, 2, 2048, 64, 8, 512
    inp, out = _moe16_case(qg, fmt, M, H, E, topk, I, seed=1688)
    W = {k: dev(v) for k, v in inp.items()}
    ids8 = torch.empty((M, topk), dtype=torch.int32, device="cuda")
    y8 = host(qg.qg_moe_ffn(fmt, W["x"], W["Wr"], topk, W["Wg"], W["Wu"], W["Wd"], W["sg"], W["su"], W["sd"], I,
                            topk_ids=ids8))
    np.testing.assert_array_equal(host(ids8), out["ids"])
    y_exact = _moe_exact(inp, fmt, out["ids"], out["w"].astype(np.float64), topk, I)
    e16 = np.abs(out["y"] - y_exact).max()
    e8 = np.abs(y8 - y_exact).max()
    print(f"max |y - y_exact|: s16 {e16:.3e}, int8 {e8:.3e}")
    assert e16 * 20 < e8


def test_no_device_error_recorded(qg):
    assert qg.qg_device_error() == 0
