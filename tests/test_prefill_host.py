"""The prefill GEMM's tensor-core descriptors, operand swizzle and launch plans, checked on
the CPU before any GPU run (tests/prefill_model.cu, compiled with the CUDA compiler for the
host side only): descriptor fields against the documented bit positions, the swizzle rule
shared by the two operand producers, and for every CTA of the planned launches over a sweep
of shapes and all twelve formats the copy, output and weight-fetch ranges and alignments."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_prefill_model(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = os.path.join(str(tmp_path), "prefill_model")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a", "--expt-relaxed-constexpr",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "gguf_block_quantized_quant_gb300", "csrc"),
                    os.path.join(HERE, "prefill_model.cu"), "-o", exe], check=True, capture_output=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0 and "fails 0" in out.stdout, out.stdout[-3000:]
