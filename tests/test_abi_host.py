"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/qg.h declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qg.h")


@pytest.fixture(scope="module")
def L():
    from gguf_block_quantized_quant_gb300 import build
    build.build()
    import gguf_block_quantized_quant_gb300 as qg
    return qg.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qg_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    import gguf_block_quantized_quant_gb300 as qg
    assert sorted(qg.EXPORTS) == _declared_functions()


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_library_targets_sm103a_only():
    from gguf_block_quantized_quant_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version_and_strerror(L):
    import gguf_block_quantized_quant_gb300 as qg
    assert qg.qg_version() >= 100
    for st in (0, -1, -2, -3, -4, -5):
        assert qg.strerror(st) and qg.strerror(st) != "unknown status"


def _P(v):
    return ctypes.c_void_p(v)


A16 = 0x10000     # fake, never dereferenced: argument checks fail before any device use


def test_gemv_rejects_bad_arguments(L):
    L_ = L
    ok = dict(fmt=12, W=A16, x=A16, y=A16, N=4, K=256, M=1)

    def call(**kw):
        a = dict(ok, **kw)
        return L_.qg_gemv(a["fmt"], _P(a["W"]), _P(a["x"]), _P(a["y"]), a["N"], a["K"], a["M"], None, 0, None)

    assert call(fmt=5) == -1          # unknown format (type id 5 is unused)
    assert call(K=255) == -1          # not a multiple of the block size
    assert call(K=0) == -1
    assert call(M=0) == -1
    assert call(M=17) == -1           # batch above 16
    assert call(N=0) == -1
    assert call(W=0) == -1            # null pointer
    assert call(x=0) == -1
    assert call(W=A16 + 8) == -3      # weights not 16-byte aligned
    assert call(y=A16 + 2) == -3
    assert call() == -2               # valid arguments but no workspace


def test_other_entry_points_reject_bad_arguments(L):
    P = _P
    assert L.qg_quantize_act(P(A16), 1, 33, P(A16), P(A16), P(A16), None) == -1
    assert L.qg_gemv_q(12, P(A16), None, P(A16), P(A16), P(A16), 4, 256, 1, None, 0, None) == -1
    assert L.qg_gemv_static_ws(5, P(A16), P(A16), P(A16), 4, 256, 1, None) == -1    # unknown format
    assert L.qg_gemv_static_ws(12, P(A16), None, P(A16), 4, 256, 1, None) == -1     # no activations
    assert L.qg_gemv_static_ws(12, P(A16), P(A16), P(A16), 4, 256, 17, None) == -1  # batch above 16
    assert L.qg_block_dots(14, P(A16), P(A16), P(A16 + 2), 4, 256, 1, P(A16), P(A16), None) == -3
    args = [12, P(A16), 1, 2048, P(A16), 256, 8] + [P(A16)] * 6 + [512, P(A16), None, None]
    assert L.qg_moe_ffn(*args, None, 0, None) == -2                      # no workspace
    bad_topk = list(args)
    bad_topk[6] = 17
    assert L.qg_moe_ffn(*bad_topk, P(A16), 1 << 30, None) == -1
    assert L.qg_moe_ffn_s16(*args, None, 0, None) == -2                  # no workspace
    assert L.qg_moe_ffn_s16(*bad_topk, P(A16), 1 << 30, None) == -1
    assert L.qg_quantize_act_s16(P(A16), 1, 33, P(A16), P(A16), P(A16), None) == -1
    assert L.qg_quantize_act_s16(P(A16), 1, 64, P(A16 + 1), P(A16), P(A16), None) == -3  # int16 codes misaligned
    assert L.qg_ffn_sublayer(12, P(A16), P(A16), P(A16), P(A16), P(A16), 1, 5120, 17408, None, 0, None) == -2
    assert L.qg_ffn_sublayer(12, P(A16), P(A16), P(A16), P(A16), P(A16), 1, 5000, 17408, P(A16), 1 << 30,
                             None) == -1


def test_workspace_sizes(L):
    import gguf_block_quantized_quant_gb300 as qg
    bad = qg.WS_INVALID
    assert qg.qg_workspace_size(qg.QG_OP_GEMV, 12, 1, 17408, 5120) != bad
    assert qg.qg_workspace_size(qg.QG_OP_GEMV, 12, 1, 17408, 5000) == bad
    assert qg.qg_workspace_size(99, 12, 1, 16, 256) == bad
    # small N is split along K: the partial sums need workspace
    assert qg.qg_workspace_size(qg.QG_OP_GEMV_Q, 12, 1, 1, 4096) >= 4 * 2
    moe = qg.qg_workspace_size(qg.QG_OP_MOE_FFN, 12, 4, 2048, 2048, 256, 8, 512)
    assert moe != bad and moe > 3 * 4 * 4 * 9 * 512
    off = qg.qg_moe_ws_layout(4, 2048, 256, 8, 512)
    assert off == sorted(off) and off[-1] < moe
    # s16: two planes of g and u per row, int16 codes of h, two image rows per activation row
    moe16 = qg.qg_workspace_size(qg.QG_OP_MOE_FFN_S16, 12, 4, 2048, 2048, 256, 8, 512)
    assert moe16 != bad and moe16 > moe
    off16 = qg.qg_moe_s16_ws_layout(4, 2048, 256, 8, 512)
    R, I = 4 * 9, 512
    assert off16 == sorted(off16) and off16[-1] < moe16
    assert off16[1] - off16[0] >= 4 * R * 2 * I and off16[3] - off16[2] >= 4 * R * I
    assert off16[4] - off16[3] >= 2 * R * I
    assert qg.qg_workspace_size(qg.QG_OP_MOE_FFN_S16, 12, 17, 2048, 2048, 256, 8, 512) == bad
    ffn = qg.qg_workspace_size(qg.QG_OP_FFN_SUBLAYER, 14, 16, 5120, 5120, 0, 0, 17408)
    assert ffn != bad and ffn >= 3 * 4 * 16 * 17408
    assert qg.qg_ffn_ws_layout(14, 16, 5120, 17408)[2] < ffn


def test_binding_takes_device_or_page_locked_tensors_only():
    """Activations may be page-locked host tensors (the kernels address them directly);
    plain pageable host tensors, and host tensors for weights or workspaces, are refused
    before any call reaches the library."""
    import torch

    import gguf_block_quantized_quant_gb300 as qg
    t = torch.zeros(16, dtype=torch.float32)
    with pytest.raises(ValueError):
        qg._ptr(t)                 # pageable host memory
    with pytest.raises(ValueError):
        qg._ptr(t, False)          # weights / workspace must be device memory
    assert qg._ptr(None) is None
