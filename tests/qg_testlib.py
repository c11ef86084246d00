"""Helpers shared by the GPU parity tests (not collected as tests)."""
import numpy as np
import pytest

import synth

FMTS = [synth.Q4_0, synth.Q4_1, synth.Q5_0, synth.Q5_1, synth.Q8_0, synth.Q2_K, synth.Q3_K, synth.Q4_K, synth.Q5_K,
        synth.Q6_K, synth.IQ4_NL, synth.IQ4_XS]
FMT_IDS = [synth.FORMAT_NAMES[f] for f in FMTS]

# Per-element bound on the final fp32 outputs against the fp64 oracle:
#   |y - y_ref| <= RTOL * sum_k |w_k * xhat_k| + ATOL
RTOL, ATOL = 1e-5, 1e-6


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def qg_module():
    torch_cuda()
    import gguf_block_quantized_quant_gb300 as qg
    from gguf_block_quantized_quant_gb300 import build
    build.build()
    return qg


def dev(a):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_within(y, y_ref, sabs, what, rtol=RTOL, atol=ATOL):
    y = np.asarray(y, np.float64)
    err = np.abs(y - y_ref)
    bound = rtol * sabs + atol
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of bound; worst at {i}: "
                             f"got {y[i]!r} want {y_ref[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    return float((err / bound).max()) if err.size else 0.0
