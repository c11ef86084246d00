"""CPU oracle for the quantized GEMV / MoE FFN / FFN sublayer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``gguf_block_quantized_quant_gb300``) never imports it and shares no code with it.

This module compiles ``qg_oracle.c`` with the host C compiler into
``oracle/_build/liboracle.so`` and exposes numpy-friendly wrappers.  The C file
is the oracle; this file only marshals arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qg_oracle.c")
_HDR = os.path.join(_HERE, "qg_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K, IQ4_NL, IQ4_XS = 2, 3, 6, 7, 8, 12, 13, 14, 20, 23
Q2_K, Q3_K = 10, 11
FORMATS = {"Q4_0": Q4_0, "Q4_1": Q4_1, "Q5_0": Q5_0, "Q5_1": Q5_1, "Q8_0": Q8_0, "Q2_K": Q2_K, "Q3_K": Q3_K,
           "Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K, "IQ4_NL": IQ4_NL, "IQ4_XS": IQ4_XS}
_QK = {Q4_0: 32, Q4_1: 32, Q5_0: 32, Q5_1: 32, Q8_0: 32, Q2_K: 256, Q3_K: 256, Q4_K: 256, Q5_K: 256, Q6_K: 256,
       IQ4_NL: 32, IQ4_XS: 256}
_BS = {Q4_0: 18, Q4_1: 20, Q5_0: 22, Q5_1: 24, Q8_0: 34, Q2_K: 84, Q3_K: 110, Q4_K: 144, Q5_K: 176, Q6_K: 210,
       IQ4_NL: 18, IQ4_XS: 136}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, OpenMP).  Returns the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(L):
    P = ctypes.c_void_p
    i = ctypes.c_int
    L.or_block_elems.argtypes = [i]
    L.or_block_bytes.argtypes = [i]
    L.or_half_to_double.argtypes = [ctypes.c_uint16]
    L.or_half_to_double.restype = ctypes.c_double
    L.or_decode_block.argtypes = [i, P, P, P, P, P]
    L.or_decode_block_mc.argtypes = [i, P, P, P, P, P, P]
    L.or_dequant_matrix.argtypes = [i, P, i, i, P]
    L.or_quantize_act.argtypes = [P, i, i, P, P, P]
    L.or_block_dots.argtypes = [i, P, P, P, i, i, i, P, P]
    L.or_gemv_q.argtypes = [i, P, P, P, P, i, i, i, P]
    L.or_gemv_deq.argtypes = [i, P, P, P, i, i, i, P]
    L.or_absdot.argtypes = [i, P, P, P, i, i, i, P]
    L.or_gemv.argtypes = [i, P, P, i, i, i, P]
    L.or_router.argtypes = [P, i, i, P, i, i, P, P, P, P]
    L.or_swiglu.argtypes = [ctypes.c_double, ctypes.c_double]
    L.or_swiglu.restype = ctypes.c_double
    L.or_moe_gateup.argtypes = [i, P, i, i, i, i, i, P, P, P, P, P, P, P, P]
    L.or_requant.argtypes = [P, i, i, P, P, P]
    L.or_moe_down.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P, P, P]
    L.or_moe_ffn.argtypes = [i, P, i, i, P, i, i, P, P, P, P, P, P, i, P, P, P]
    L.or_ffn_sublayer.argtypes = [i, P, P, P, P, i, i, i, P, P, P, P]
    L.or_quantize_act16.argtypes = [P, i, i, P, P, P]
    L.or_gemv_q16.argtypes = [i, P, P, P, P, i, i, i, P]
    L.or_absdot16.argtypes = [i, P, P, P, i, i, i, P]
    L.or_moe_gateup16.argtypes = [i, P, i, i, i, i, i, P, P, P, P, P, P, P, P]
    L.or_requant16.argtypes = [P, i, i, P, P, P]
    L.or_moe_down16.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P, P, P]
    L.or_moe_ffn16.argtypes = [i, P, i, i, P, i, i, P, P, P, P, P, P, i, P, P, P]
    L.or_float_to_half.argtypes = [ctypes.c_float]
    L.or_float_to_half.restype = ctypes.c_uint16
    L.or_float_to_half_array.argtypes = [P, ctypes.c_size_t, P]
    L.or_dequant_f16.argtypes = [i, P, i, i, P]
    L.or_prefill_gemm.argtypes = [i, P, P, i, i, i, P, P]
    L.or_set_threads.argtypes = [i]
    L.or_get_threads.restype = i
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


class use_library:
    """Context manager that points the wrappers at another build of the oracle
    (used by the tests that plant mistakes in a copy of the oracle source)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        _lib = _configure(ctypes.CDLL(self.path))
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def build_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (test use only)."""
    d = os.path.dirname(out_path)
    c = os.path.join(d, "variant.c")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["cp", _HDR, os.path.join(d, "qg_oracle.h")], check=True)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", out_path, c, "-lm"],
                   check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def block_elems(fmt):
    return _QK[fmt]


def block_bytes(fmt):
    return _BS[fmt]


def row_bytes(fmt, K):
    return (K // _QK[fmt]) * _BS[fmt]


def set_threads(n: int):
    lib().or_set_threads(int(n))


def get_threads() -> int:
    return int(lib().or_get_threads())


def half_to_double(bits: int) -> float:
    return float(lib().or_half_to_double(int(bits)))


def decode_block(fmt, blk, with_mc: bool = False):
    """Returns (w fp64[QK], codes int32[QK], A fp64[QK/32], B fp64[QK/32]), and the min
    codes int32[QK] as a fifth item when with_mc."""
    blk = _u8(blk)
    assert blk.size == _BS[fmt]
    qk = _QK[fmt]
    w = np.zeros(qk, np.float64)
    c = np.zeros(qk, np.int32)
    mc = np.zeros(qk, np.int32)
    A = np.zeros(qk // 32, np.float64)
    B = np.zeros(qk // 32, np.float64)
    lib().or_decode_block_mc(fmt, _p(blk), _p(w), _p(c), _p(mc), _p(A), _p(B))
    return (w, c, A, B, mc) if with_mc else (w, c, A, B)


def dequant_matrix(fmt, W, N, K):
    W = _u8(W)
    out = np.zeros((N, K), np.float64)
    lib().or_dequant_matrix(fmt, _p(W), N, K, _p(out))
    return out


def quantize_act(x):
    x = _f32(x)
    M, K = x.shape
    xq = np.zeros((M, K), np.int8)
    xd = np.zeros((M, K // 32), np.float32)
    xs = np.zeros((M, K // 32), np.int32)
    lib().or_quantize_act(_p(x), M, K, _p(xq), _p(xd), _p(xs))
    return xq, xd, xs


def block_dots(fmt, W, xq, xs, N, K):
    W = _u8(W)
    xq = np.ascontiguousarray(xq, np.int8)
    xs = np.ascontiguousarray(xs, np.int32)
    M = xq.shape[0]
    dots = np.zeros((M, N, K // 32), np.int32)
    aux = np.zeros((M, N, K // 32), np.int32)
    lib().or_block_dots(fmt, _p(W), _p(xq), _p(xs), N, K, M, _p(dots), _p(aux))
    return dots, aux


def gemv_q(fmt, W, xq, xd, xs, N, K):
    W = _u8(W)
    xq = np.ascontiguousarray(xq, np.int8)
    xd = _f32(xd)
    xs = np.ascontiguousarray(xs, np.int32)
    M = xq.shape[0]
    y = np.zeros((M, N), np.float64)
    lib().or_gemv_q(fmt, _p(W), _p(xq), _p(xd), _p(xs), N, K, M, _p(y))
    return y


def gemv_deq(fmt, W, xq, xd, N, K):
    W = _u8(W)
    xq = np.ascontiguousarray(xq, np.int8)
    xd = _f32(xd)
    M = xq.shape[0]
    y = np.zeros((M, N), np.float64)
    lib().or_gemv_deq(fmt, _p(W), _p(xq), _p(xd), N, K, M, _p(y))
    return y


def absdot(fmt, W, xq, xd, N, K):
    W = _u8(W)
    xq = np.ascontiguousarray(xq, np.int8)
    xd = _f32(xd)
    M = xq.shape[0]
    s = np.zeros((M, N), np.float64)
    lib().or_absdot(fmt, _p(W), _p(xq), _p(xd), N, K, M, _p(s))
    return s


def gemv(fmt, W, x, N, K):
    W = _u8(W)
    x = _f32(x)
    M = x.shape[0]
    y = np.zeros((M, N), np.float64)
    lib().or_gemv(fmt, _p(W), _p(x), N, K, M, _p(y))
    return y


def router(x, Wr, topk):
    x = _f32(x)
    Wr = _f32(Wr)
    M, H = x.shape
    E = Wr.shape[0]
    logits = np.zeros((M, E), np.float64)
    probs = np.zeros((M, E), np.float64)
    ids = np.zeros((M, topk), np.int32)
    w = np.zeros((M, topk), np.float64)
    lib().or_router(_p(x), M, H, _p(Wr), E, topk, _p(logits), _p(probs), _p(ids), _p(w))
    return logits, probs, ids, w


def swiglu(g, u):
    return float(lib().or_swiglu(float(g), float(u)))


def moe_gateup(fmt, x, E, topk, I, ids, Wg_exps, Wu_exps, Wg_sh, Wu_sh):
    x = _f32(x)
    M, H = x.shape
    ids = np.ascontiguousarray(ids, np.int32)
    S = topk + 1
    g = np.zeros((M, S, I), np.float64)
    u = np.zeros((M, S, I), np.float64)
    h = np.zeros((M, S, I), np.float64)
    lib().or_moe_gateup(fmt, _p(x), M, H, E, topk, I, _p(ids), _p(_u8(Wg_exps)), _p(_u8(Wu_exps)),
                        _p(_u8(Wg_sh)), _p(_u8(Wu_sh)), _p(g), _p(u), _p(h))
    return g, u, h


def requant(h):
    h = np.ascontiguousarray(h, np.float64)
    R, I = h.shape
    hq = np.zeros((R, I), np.int8)
    hd = np.zeros((R, I // 32), np.float32)
    hs = np.zeros((R, I // 32), np.int32)
    lib().or_requant(_p(h), R, I, _p(hq), _p(hd), _p(hs))
    return hq, hd, hs


def moe_down(fmt, M, H, E, topk, I, ids, w, hq, hd, hs, Wd_exps, Wd_sh, want_o=False):
    S = topk + 1
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    hq = np.ascontiguousarray(hq, np.int8).reshape(M * S, I)
    hd = _f32(hd).reshape(M * S, I // 32)
    hs = np.ascontiguousarray(hs, np.int32).reshape(M * S, I // 32)
    y = np.zeros((M, H), np.float64)
    yabs = np.zeros((M, H), np.float64)
    o = np.zeros((M, S, H), np.float64) if want_o else None
    lib().or_moe_down(fmt, M, H, E, topk, I, _p(ids), _p(w), _p(hq), _p(hd), _p(hs),
                      _p(_u8(Wd_exps)), _p(_u8(Wd_sh)), _p(y), _p(o), _p(yabs))
    return (y, yabs, o) if want_o else (y, yabs)


def moe_ffn(fmt, x, Wr, topk, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I):
    x = _f32(x)
    Wr = _f32(Wr)
    M, H = x.shape
    E = Wr.shape[0]
    y = np.zeros((M, H), np.float64)
    ids = np.zeros((M, topk), np.int32)
    w = np.zeros((M, topk), np.float64)
    lib().or_moe_ffn(fmt, _p(x), M, H, _p(Wr), E, topk, _p(_u8(Wg_exps)), _p(_u8(Wu_exps)),
                     _p(_u8(Wd_exps)), _p(_u8(Wg_sh)), _p(_u8(Wu_sh)), _p(_u8(Wd_sh)), I,
                     _p(y), _p(ids), _p(w))
    return y, ids, w


def ffn_sublayer(fmt, Wg, Wu, Wd, x, I):
    x = _f32(x)
    M, H = x.shape
    y = np.zeros((M, H), np.float64)
    g = np.zeros((M, I), np.float64)
    u = np.zeros((M, I), np.float64)
    h = np.zeros((M, I), np.float64)
    lib().or_ffn_sublayer(fmt, _p(_u8(Wg)), _p(_u8(Wu)), _p(_u8(Wd)), _p(x), M, H, I,
                          _p(y), _p(g), _p(u), _p(h))
    return y, g, u, h


# ----------------------------------------------------------------------------- s16 activations
def quantize_act16(x):
    x = _f32(x)
    M, K = x.shape
    xq = np.zeros((M, K), np.int16)
    xd = np.zeros((M, K // 32), np.float32)
    xs = np.zeros((M, K // 32), np.int32)
    lib().or_quantize_act16(_p(x), M, K, _p(xq), _p(xd), _p(xs))
    return xq, xd, xs


def gemv_q16(fmt, W, xq, xd, xs, N, K):
    W = _u8(W)
    xq = np.ascontiguousarray(xq, np.int16)
    xd = _f32(xd)
    xs = np.ascontiguousarray(xs, np.int32)
    M = xq.shape[0]
    y = np.zeros((M, N), np.float64)
    lib().or_gemv_q16(fmt, _p(W), _p(xq), _p(xd), _p(xs), N, K, M, _p(y))
    return y


def absdot16(fmt, W, xq, xd, N, K):
    W = _u8(W)
    xq = np.ascontiguousarray(xq, np.int16)
    xd = _f32(xd)
    M = xq.shape[0]
    s = np.zeros((M, N), np.float64)
    lib().or_absdot16(fmt, _p(W), _p(xq), _p(xd), N, K, M, _p(s))
    return s


def moe_gateup16(fmt, x, E, topk, I, ids, Wg_exps, Wu_exps, Wg_sh, Wu_sh):
    x = _f32(x)
    M, H = x.shape
    ids = np.ascontiguousarray(ids, np.int32)
    S = topk + 1
    g = np.zeros((M, S, I), np.float64)
    u = np.zeros((M, S, I), np.float64)
    h = np.zeros((M, S, I), np.float64)
    lib().or_moe_gateup16(fmt, _p(x), M, H, E, topk, I, _p(ids), _p(_u8(Wg_exps)), _p(_u8(Wu_exps)),
                          _p(_u8(Wg_sh)), _p(_u8(Wu_sh)), _p(g), _p(u), _p(h))
    return g, u, h


def requant16(h):
    h = np.ascontiguousarray(h, np.float64)
    R, I = h.shape
    hq = np.zeros((R, I), np.int16)
    hd = np.zeros((R, I // 32), np.float32)
    hs = np.zeros((R, I // 32), np.int32)
    lib().or_requant16(_p(h), R, I, _p(hq), _p(hd), _p(hs))
    return hq, hd, hs


def moe_down16(fmt, M, H, E, topk, I, ids, w, hq, hd, hs, Wd_exps, Wd_sh, want_o=False):
    S = topk + 1
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    hq = np.ascontiguousarray(hq, np.int16).reshape(M * S, I)
    hd = _f32(hd).reshape(M * S, I // 32)
    hs = np.ascontiguousarray(hs, np.int32).reshape(M * S, I // 32)
    y = np.zeros((M, H), np.float64)
    yabs = np.zeros((M, H), np.float64)
    o = np.zeros((M, S, H), np.float64) if want_o else None
    lib().or_moe_down16(fmt, M, H, E, topk, I, _p(ids), _p(w), _p(hq), _p(hd), _p(hs),
                        _p(_u8(Wd_exps)), _p(_u8(Wd_sh)), _p(y), _p(o), _p(yabs))
    return (y, yabs, o) if want_o else (y, yabs)


def moe_ffn16(fmt, x, Wr, topk, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I):
    x = _f32(x)
    Wr = _f32(Wr)
    M, H = x.shape
    E = Wr.shape[0]
    y = np.zeros((M, H), np.float64)
    ids = np.zeros((M, topk), np.int32)
    w = np.zeros((M, topk), np.float64)
    lib().or_moe_ffn16(fmt, _p(x), M, H, _p(Wr), E, topk, _p(_u8(Wg_exps)), _p(_u8(Wu_exps)),
                       _p(_u8(Wd_exps)), _p(_u8(Wg_sh)), _p(_u8(Wu_sh)), _p(_u8(Wd_sh)), I,
                       _p(y), _p(ids), _p(w))
    return y, ids, w


# ----------------------------------------------------------------------------- prefill (fp16 operands)
def float_to_half(x):
    """fp32 -> fp16 bit patterns (uint16), round to nearest, ties to even."""
    x = _f32(x)
    out = np.zeros(x.shape, np.uint16)
    lib().or_float_to_half_array(_p(x), x.size, _p(out))
    return out


def dequant_f16(fmt, W, N, K):
    """The fp16 weights (bit patterns, N x K uint16) of the prefill reading."""
    W = _u8(W)
    out = np.zeros((N, K), np.uint16)
    lib().or_dequant_f16(fmt, _p(W), N, K, _p(out))
    return out


def prefill_gemm(fmt, W, x, N, K):
    """y[m][n] = sum_k w16[n][k] * x16[m][k] in fp64; returns (y, sabs), both M x N."""
    x = _f32(x)
    M = x.shape[0]
    assert x.shape[1] == K
    y = np.zeros((M, N), np.float64)
    sabs = np.zeros((M, N), np.float64)
    lib().or_prefill_gemm(fmt, _p(_u8(W)), _p(x), N, K, M, _p(y), _p(sabs))
    return y, sabs
