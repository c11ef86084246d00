"""The oracle's pins must catch plausible mistakes.

Each case edits one line of a copy of the oracle source (a dropped term, a wrong
sign, a wrong or transposed index, the wrong rounding mode), compiles the copy on
the CPU, and runs the pin tests against it: at least one pin must fail.  Nothing
here touches the real oracle build or any GPU.
"""
import os

import pytest

import oracle
import test_oracle_pins as pins

# (name, original text, mutated text)
MUTATIONS = [
    ("q4_0 offset", "code = nib - 8;", "code = nib - 7;"),
    ("q8_0 scale field", "a = rd_half(blk);\n            code = (int8_t)blk[2 + e];",
     "a = rd_half(blk + 1);\n            code = (int8_t)blk[2 + e];"),
    ("q4_k high scale bits", "((sc12[j - 4] >> 6) << 4)", "((sc12[j - 4] >> 6) << 3)"),
    ("q4_k min bits from wrong byte", "((sc12[j] >> 6) << 4)", "((sc12[j - 4] >> 6) << 4)"),
    ("k-quant min term dropped", "b = dmin * M;", "b = 0;"),
    ("k-quant nibble half swapped", "(j % 2 == 0) ? (byte & 15) : (byte >> 4)",
     "(j % 2 == 1) ? (byte & 15) : (byte >> 4)"),
    ("q5_k qh index transposed", "((qh[l] >> j) & 1)", "((qh[j] >> l) & 1)"),
    ("q6_k ql half", "32 * (t & 1)", "32 * (t >> 1)"),
    ("q6_k qh shift", "(2 * t)) & 3", "(t)) & 3"),
    ("q6_k scale index", "sc[e / 16]", "sc[e / 32]"),
    ("iq4 nibble order", "(j < 16) ? (byte & 15) : (byte >> 4)", "(j < 16) ? (byte >> 4) : (byte & 15)"),
    ("iq4 scale offset", "a = d * (ls - 32);", "a = d * (ls - 31);"),
    ("quant rounding mode", "q = (int)roundf(v);", "q = (int)rintf(v);"),
    ("quant reciprocal", "float v = xb[i] / d;", "float v = xb[i] * (1.0f / d);"),
    ("gemv min sign", "- B[ub] * s_x", "+ B[ub] * s_x"),
    ("router tie order", "p[e] > p[best]", "p[e] >= p[best]"),
    ("router no renorm", "w[(size_t)m * topk + s] /= wsum;", "w[(size_t)m * topk + s] /= 1.0;"),
    ("swiglu sign", "1.0 + exp(-g)", "1.0 + exp(g)"),
    ("shared expert weighted", "double ws = s < topk ? w[(size_t)m * topk + s] : 1.0;",
     "double ws = s < topk ? w[(size_t)m * topk + s] : 0.5;"),
    ("fp16 exponent bias", "expo - 25", "expo - 24"),
    ("q4_1 min sign", "b = -rd_half(blk + 2);\n            code = e < 16", "b = rd_half(blk + 2);\n            code = e < 16"),
    ("q5 fifth bit index", "int hb = (qh[e / 8] >> (e % 8)) & 1;", "int hb = (qh[e / 8] >> (e % 4)) & 1;"),
    ("q5_0 offset dropped", "else code -= 16;", "else code -= 0;"),
    ("q5_1 min from wrong field", "if (one) b = -rd_half(blk + 2);", "if (one) b = -rd_half(blk + 4);"),
    ("iq4_nl nibble order", "int idx = e < 16 ? (blk[2 + e] & 15) : (blk[2 + e - 16] >> 4);",
     "int idx = e < 16 ? (blk[2 + e] >> 4) : (blk[2 + e - 16] & 15);"),
    ("q2_k scale and min nibbles swapped", "code = (blk[sb] & 15) * q2;\n                mcode = blk[sb] >> 4;",
     "code = (blk[sb] >> 4) * q2;\n                mcode = blk[sb] & 15;"),
    ("q2_k dmin field", "b = rd_half(blk + 82);", "b = rd_half(blk + 80);"),
    ("q2_k code shift", "int q2 = (blk[16 + 32 * h + l] >> (2 * j)) & 3;", "int q2 = (blk[16 + 32 * h + l] >> j) & 3;"),
    ("q2_k dots aux from the plain sum", "int32_t a = fmt == OR_Q2_K ? msum", "int32_t a = fmt == OR_Q3_K ? msum"),
    ("q2_k gemv min from the plain sum", "double s_x = fmt == OR_Q2_K ? (double)msum",
     "double s_x = fmt == OR_Q3_K ? (double)msum"),
    ("q3_k high-bit index transposed", "int hb = (blk[l] >> (4 * h + j)) & 1;", "int hb = (blk[l] >> (4 * j + h)) & 1;"),
    ("q3_k offset on the wrong bit value", "(q2 - (hb ? 0 : 4))", "(q2 - (hb ? 4 : 0))"),
    ("q3_k scale high bits transposed", "int high2 = (sc12[8 + i % 4] >> (2 * (i / 4))) & 3;",
     "int high2 = (sc12[8 + i / 4] >> (2 * (i % 4))) & 3;"),
    ("q3_k scale offset", "return (low4 | (high2 << 4)) - 32;", "return (low4 | (high2 << 4)) - 31;"),
    ("s16 step", "quantize_rows(x, M, K, 32512.0f, NULL, xq, xd, xs);",
     "quantize_rows(x, M, K, 32767.0f, NULL, xq, xd, xs);"),
    ("s16 codes narrowed to a byte", "return a.q8 ? (int32_t)a.q8[i] : (int32_t)a.q16[i];",
     "return a.q8 ? (int32_t)a.q8[i] : (int32_t)(int8_t)a.q16[i];"),
    ("moe s16 gate/up input at the int8 step", "bits == 8 ? 127.0f : 32512.0f, q8, q16, xd, xs);",
     "127.0f, q8, q16, xd, xs);"),
    ("moe s16 h requantized at the int8 step", "quantize_rows(hf, (int)R, I, bits == 8 ? 127.0f : 32512.0f,",
     "quantize_rows(hf, (int)R, I, 127.0f,"),
    ("fp16 ties away from zero", "if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;",
     "if (frac >= 0.5) r += 1.0;"),
    ("fp16 no gradual underflow", "if (e < -14) e = -14;", "if (e < -15) e = -15;"),
    ("fp16 overflow threshold", "if (e > 15) return (uint16_t)(sign | 0x7c00u);",
     "if (e > 16) return (uint16_t)(sign | 0x7c00u);"),
    ("prefill weight min term dropped", "float w32 = p1 - p2;", "float w32 = p1;"),
    ("prefill activation not rounded to fp16", "x16[i] = or_half_to_double(or_float_to_half(x[i]));",
     "x16[i] = (double)x[i];"),
    ("prefill rows reversed", "dequant_row_f16(fmt, W + (size_t)n * rb, K, w16);",
     "dequant_row_f16(fmt, W + (size_t)(N - 1 - n) * rb, K, w16);"),
]

PIN_TESTS = [name for name in dir(pins) if name.startswith("test_")]


def _run_pins(orc):
    """Run every pin (all parametrizations); return the names of those that failed."""
    failed = []
    for name in PIN_TESTS:
        fn = getattr(pins, name)
        params = [None]
        if "fmt" in fn.__code__.co_varnames[:fn.__code__.co_argcount]:
            params = pins.FMTS
        for p in params:
            try:
                fn(orc, p) if p is not None else fn(orc)
            except (AssertionError, ValueError, IndexError, OverflowError):
                failed.append(f"{name}[{p}]")
            except Exception as exc:  # noqa: BLE001 - any exception is a caught mistake
                failed.append(f"{name}[{p}]:{type(exc).__name__}")
    return failed


@pytest.mark.parametrize("name,orig,mut", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, orig, mut):
    src = oracle.source_text()
    assert src.count(orig) >= 1, f"mutation anchor not found: {orig!r}"
    path = oracle.build_variant(src.replace(orig, mut, 1), os.path.join(str(tmp_path), "libvariant.so"))
    with oracle.use_library(path):
        failed = _run_pins(oracle)
    assert failed, f"no pin caught the planted mistake '{name}'"


def test_unmutated_copy_passes(tmp_path):
    path = oracle.build_variant(oracle.source_text(), os.path.join(str(tmp_path), "libvariant.so"))
    with oracle.use_library(path):
        assert _run_pins(oracle) == []
