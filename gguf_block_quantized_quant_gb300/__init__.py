"""Python binding of libqg: decode GEMV on raw GGUF blocks for GB300 (sm_103a).

Thin marshalling layer over the C ABI declared in ``include/qg.h``: every function here
has the name of the C entry point it calls, takes torch CUDA tensors, passes their device
pointers and the current CUDA stream, and raises ``QGError`` on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; PyTorch only provides device memory and
streams.  If ``libqg.so`` has not been built, every call raises: there is no fallback.

Block formats (GGUF type ids): Q4_0=2, Q4_1=3, Q5_0=6, Q5_1=7, Q8_0=8, Q2_K=10, Q3_K=11,
Q4_K=12, Q5_K=13, Q6_K=14, IQ4_NL=20, IQ4_XS=23.
A weight matrix of N rows and K columns is passed as a uint8 CUDA tensor holding the N
rows of raw blocks back to back (``row_bytes(fmt, K)`` bytes per row).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K, IQ4_NL, IQ4_XS = 2, 3, 6, 7, 8, 12, 13, 14, 20, 23
Q2_K, Q3_K = 10, 11
FORMATS = {"Q4_0": Q4_0, "Q4_1": Q4_1, "Q5_0": Q5_0, "Q5_1": Q5_1, "Q8_0": Q8_0, "Q2_K": Q2_K, "Q3_K": Q3_K,
           "Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K, "IQ4_NL": IQ4_NL, "IQ4_XS": IQ4_XS}
BLOCK_ELEMS = {Q4_0: 32, Q4_1: 32, Q5_0: 32, Q5_1: 32, Q8_0: 32, Q2_K: 256, Q3_K: 256, Q4_K: 256, Q5_K: 256,
               Q6_K: 256, IQ4_NL: 32, IQ4_XS: 256}
BLOCK_BYTES = {Q4_0: 18, Q4_1: 20, Q5_0: 22, Q5_1: 24, Q8_0: 34, Q2_K: 84, Q3_K: 110, Q4_K: 144, Q5_K: 176,
               Q6_K: 210, IQ4_NL: 18, IQ4_XS: 136}

QG_OP_GEMV, QG_OP_GEMV_Q, QG_OP_MOE_FFN, QG_OP_FFN_SUBLAYER, QG_OP_MOE_FFN_S16, QG_OP_PREFILL = 1, 2, 3, 4, 5, 6
QG_OK, QG_EINVAL, QG_EWORKSPACE, QG_EALIGN, QG_ECUDA, QG_EDEVICE = 0, -1, -2, -3, -4, -5
WS_INVALID = ctypes.c_size_t(-1).value

LIB_PATH = _build.LIB

# every symbol declared in include/qg.h
EXPORTS = ("qg_quantize_act", "qg_gemv", "qg_gemv_q", "qg_moe_ffn", "qg_ffn_sublayer", "qg_workspace_size",
           "qg_moe_ws_layout", "qg_ffn_ws_layout", "qg_block_dots", "qg_device_error", "qg_strerror",
           "qg_version", "qg_gemv_static_ws", "qg_quantize_act_s16", "qg_moe_ffn_s16", "qg_moe_s16_ws_layout",
           "qg_prefill_gemm", "qg_dequant_f16", "qg_test_wait_expiry")
QG_STATIC_WS_BYTES = 2097152  # include/qg.h


class QGError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: status {status} ({strerror(status)})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if libqg.so is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libqg.so not found at {LIB_PATH}; build it first "
                "(python -c 'import __graft_entry__ as g; g.build()'). There is no CPU fallback.")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.qg_quantize_act.argtypes = [P, I, I, P, P, P, P]
        L.qg_gemv.argtypes = [I, P, P, P, I, I, I, P, S, P]
        L.qg_gemv_q.argtypes = [I, P, P, P, P, P, I, I, I, P, S, P]
        L.qg_gemv_static_ws.argtypes = [I, P, P, P, I, I, I, P]
        L.qg_moe_ffn.argtypes = [I, P, I, I, P, I, I, P, P, P, P, P, P, I, P, P, P, P, S, P]
        L.qg_moe_ffn_s16.argtypes = [I, P, I, I, P, I, I, P, P, P, P, P, P, I, P, P, P, P, S, P]
        L.qg_quantize_act_s16.argtypes = [P, I, I, P, P, P, P]
        L.qg_moe_s16_ws_layout.argtypes = [I, I, I, I, I, ctypes.POINTER(S)]
        L.qg_ffn_sublayer.argtypes = [I, P, P, P, P, P, I, I, I, P, S, P]
        L.qg_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        L.qg_workspace_size.restype = S
        L.qg_moe_ws_layout.argtypes = [I, I, I, I, I, ctypes.POINTER(S)]
        L.qg_ffn_ws_layout.argtypes = [I, I, I, I, ctypes.POINTER(S)]
        L.qg_block_dots.argtypes = [I, P, P, P, I, I, I, P, P, P]
        L.qg_prefill_gemm.argtypes = [I, P, P, P, I, I, I, P, S, P]
        L.qg_dequant_f16.argtypes = [I, P, I, I, P, P]
        L.qg_test_wait_expiry.argtypes = [ctypes.c_ulonglong, P]
        L.qg_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.qg_strerror.argtypes = [I]
        L.qg_strerror.restype = ctypes.c_char_p
        L.qg_version.restype = I
        for name in EXPORTS:
            getattr(L, name)
        _lib = L
    return _lib


def strerror(status: int) -> str:
    try:
        return lib().qg_strerror(int(status)).decode()
    except RuntimeError:
        return "libqg not loaded"


def row_bytes(fmt: int, K: int) -> int:
    return (K // BLOCK_ELEMS[fmt]) * BLOCK_BYTES[fmt]


def _ptr(t, host_ok=True):
    """Device address of a tensor: a CUDA tensor, or (where the C API allows host memory:
    activations and outputs) a page-locked host tensor, which the kernels address directly."""
    if t is None:
        return None
    if not (t.is_cuda or (host_ok and t.is_pinned())):
        raise ValueError("libqg takes CUDA tensors" + (" or page-locked (pinned) host tensors" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError("libqg takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t):
    """The CUDA device of a call whose activations are t (the current device for host t)."""
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _out(shape, dtype, like):
    """An output next to the activations: on their device, or page-locked host memory."""
    if like.is_cuda:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return torch.empty(shape, dtype=dtype, pin_memory=True)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != 0:
        raise QGError(rc, what)


def _ws(ws, size_query, like):
    """The workspace and its byte count: the caller's (the C call checks its size), or a new
    one of qg_workspace_size bytes on the device of the activations `like` (size_query()
    and the device lookup run only then)."""
    if ws is not None:
        return ws, ws.numel()
    nbytes = size_query()
    if nbytes == WS_INVALID:
        raise QGError(QG_EINVAL, "qg_workspace_size")
    if nbytes > 0:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=_dev(like))
    return ws, (0 if ws is None else ws.numel())


# ----------------------------------------------------------------------------- entry points
def qg_workspace_size(op: int, fmt: int, M: int, N: int, K: int, E: int = 0, topk: int = 0, I: int = 0) -> int:
    return int(lib().qg_workspace_size(op, fmt, M, N, K, E, topk, I))


def qg_quantize_act(x, xq=None, xd=None, xs=None, stream=None):
    M, K = x.shape
    xq = _out((M, K), torch.int8, x) if xq is None else xq
    xd = _out((M, K // 32), torch.float32, x) if xd is None else xd
    xs = _out((M, K // 32), torch.int32, x) if xs is None else xs
    _check(lib().qg_quantize_act(_ptr(x), M, K, _ptr(xq), _ptr(xd), _ptr(xs), _stream(stream)),
           "qg_quantize_act")
    return xq, xd, xs


def qg_quantize_act_s16(x, xq=None, xd=None, xs=None, stream=None):
    M, K = x.shape
    xq = _out((M, K), torch.int16, x) if xq is None else xq
    xd = _out((M, K // 32), torch.float32, x) if xd is None else xd
    xs = _out((M, K // 32), torch.int32, x) if xs is None else xs
    _check(lib().qg_quantize_act_s16(_ptr(x), M, K, _ptr(xq), _ptr(xd), _ptr(xs), _stream(stream)),
           "qg_quantize_act_s16")
    return xq, xd, xs


def qg_gemv(fmt: int, W, x, N: int, y=None, ws=None, stream=None):
    M, K = x.shape
    y = _out((M, N), torch.float32, x) if y is None else y
    ws, nws = _ws(ws, lambda: qg_workspace_size(QG_OP_GEMV, fmt, M, N, K), x)
    _check(lib().qg_gemv(fmt, _ptr(W, False), _ptr(x), _ptr(y), N, K, M, _ptr(ws, False), nws, _stream(stream)), "qg_gemv")
    return y


def qg_gemv_static_ws(fmt: int, W, x, N: int, y=None, stream=None):
    """qg_gemv on the library's fixed device scratch, for callers that cannot allocate
    device memory where they call (a plugin inside a framework whose allocator owns the
    device memory, or a path that cannot afford cudaMalloc's synchronization).  Nothing is
    allocated inside the call when y is given.  Every call on a device shares the scratch:
    calls that may overlap on the GPU must be ordered on one stream.  The first call on a
    device looks up the scratch address and should come before any stream capture."""
    M, K = x.shape
    y = _out((M, N), torch.float32, x) if y is None else y
    _check(lib().qg_gemv_static_ws(fmt, _ptr(W, False), _ptr(x), _ptr(y), N, K, M, _stream(stream)), "qg_gemv_static_ws")
    return y


def qg_gemv_q(fmt: int, W, xq, xd, xs, N: int, y=None, ws=None, stream=None):
    M, K = xq.shape
    y = _out((M, N), torch.float32, xq) if y is None else y
    ws, nws = _ws(ws, lambda: qg_workspace_size(QG_OP_GEMV_Q, fmt, M, N, K), xq)
    _check(lib().qg_gemv_q(fmt, _ptr(W, False), _ptr(xq), _ptr(xd), _ptr(xs), _ptr(y), N, K, M, _ptr(ws, False), nws,
                           _stream(stream)), "qg_gemv_q")
    return y


def qg_moe_ffn(fmt: int, x, Wr, topk: int, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I: int,
               y=None, topk_ids=None, topk_w=None, ws=None, stream=None):
    M, H = x.shape
    E = Wr.shape[0]
    y = _out((M, H), torch.float32, x) if y is None else y
    ws, nws = _ws(ws, lambda: qg_workspace_size(QG_OP_MOE_FFN, fmt, M, H, H, E, topk, I), x)
    _check(lib().qg_moe_ffn(fmt, _ptr(x), M, H, _ptr(Wr, False), E, topk, _ptr(Wg_exps, False), _ptr(Wu_exps, False), _ptr(Wd_exps, False),
                            _ptr(Wg_sh, False), _ptr(Wu_sh, False), _ptr(Wd_sh, False), I, _ptr(y), _ptr(topk_ids), _ptr(topk_w),
                            _ptr(ws, False), nws, _stream(stream)), "qg_moe_ffn")
    return y


def qg_moe_ffn_s16(fmt: int, x, Wr, topk: int, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I: int,
                   y=None, topk_ids=None, topk_w=None, ws=None, stream=None):
    M, H = x.shape
    E = Wr.shape[0]
    y = _out((M, H), torch.float32, x) if y is None else y
    ws, nws = _ws(ws, lambda: qg_workspace_size(QG_OP_MOE_FFN_S16, fmt, M, H, H, E, topk, I), x)
    _check(lib().qg_moe_ffn_s16(fmt, _ptr(x), M, H, _ptr(Wr, False), E, topk, _ptr(Wg_exps, False), _ptr(Wu_exps, False),
                                _ptr(Wd_exps, False), _ptr(Wg_sh, False), _ptr(Wu_sh, False), _ptr(Wd_sh, False), I, _ptr(y), _ptr(topk_ids),
                                _ptr(topk_w), _ptr(ws, False), nws, _stream(stream)), "qg_moe_ffn_s16")
    return y


def qg_ffn_sublayer(fmt: int, Wg, Wu, Wd, x, I: int, y=None, ws=None, stream=None):
    M, H = x.shape
    y = _out((M, H), torch.float32, x) if y is None else y
    ws, nws = _ws(ws, lambda: qg_workspace_size(QG_OP_FFN_SUBLAYER, fmt, M, H, H, 0, 0, I), x)
    _check(lib().qg_ffn_sublayer(fmt, _ptr(Wg, False), _ptr(Wu, False), _ptr(Wd, False), _ptr(x), _ptr(y), M, H, I, _ptr(ws, False), nws,
                                 _stream(stream)), "qg_ffn_sublayer")
    return y


def qg_moe_ws_layout(M: int, H: int, E: int, topk: int, I: int):
    off = (ctypes.c_size_t * 7)()
    _check(lib().qg_moe_ws_layout(M, H, E, topk, I, off), "qg_moe_ws_layout")
    return list(off)


def qg_moe_s16_ws_layout(M: int, H: int, E: int, topk: int, I: int):
    off = (ctypes.c_size_t * 7)()
    _check(lib().qg_moe_s16_ws_layout(M, H, E, topk, I, off), "qg_moe_s16_ws_layout")
    return list(off)


def qg_ffn_ws_layout(fmt: int, M: int, H: int, I: int):
    off = (ctypes.c_size_t * 3)()
    _check(lib().qg_ffn_ws_layout(fmt, M, H, I, off), "qg_ffn_ws_layout")
    return list(off)


def qg_block_dots(fmt: int, W, xq, xs, N: int, stream=None):
    M, K = xq.shape
    dots = _out((M, N, K // 32), torch.int32, xq)
    aux = _out((M, N, K // 32), torch.int32, xq)
    _check(lib().qg_block_dots(fmt, _ptr(W, False), _ptr(xq), _ptr(xs), N, K, M, _ptr(dots), _ptr(aux), _stream(stream)),
           "qg_block_dots")
    return dots, aux


def qg_prefill_gemm(fmt: int, W, x, N: int, y=None, ws=None, stream=None):
    """Prefill GEMM on the tensor cores: y = fp16(W) fp16(x)^T in fp32, for M >> 16 tokens."""
    M, K = x.shape
    y = _out((M, N), torch.float32, x) if y is None else y
    ws, nws = _ws(ws, lambda: qg_workspace_size(QG_OP_PREFILL, fmt, M, N, K), x)
    _check(lib().qg_prefill_gemm(fmt, _ptr(W, False), _ptr(x), _ptr(y), N, K, M, _ptr(ws, False), nws,
                                 _stream(stream)), "qg_prefill_gemm")
    return y


def qg_dequant_f16(fmt: int, W, N: int, K: int, stream=None):
    """Test hook: the fp16 weights (uint16 bit patterns, N x K) the prefill GEMM multiplies."""
    out = torch.empty((N, K), dtype=torch.int16, device=W.device)
    _check(lib().qg_dequant_f16(fmt, _ptr(W, False), N, K, _ptr(out), _stream(stream)), "qg_dequant_f16")
    return out


def qg_test_wait_expiry(limit_ns: int, stream=None):
    """Test hook: a bounded wait that nothing satisfies gives up after limit_ns and sets the
    device error word (read it with qg_device_error)."""
    _check(lib().qg_test_wait_expiry(int(limit_ns), _stream(stream)), "qg_test_wait_expiry")


def qg_device_error() -> int:
    v = ctypes.c_uint(0)
    _check(lib().qg_device_error(ctypes.byref(v)), "qg_device_error")
    return int(v.value)


def qg_version() -> int:
    return int(lib().qg_version())
