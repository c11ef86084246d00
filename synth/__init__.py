"""Seeded synthetic inputs shared by the tests and the benchmark.

This module only draws random bytes and numbers; it holds none of the method's
arithmetic (no decoding, quantization or dot products).  Both the CUDA path and the
CPU oracle consume the same arrays produced here.

Block formats are filled field by field: every fp16 scale field receives a value
drawn as fp32 and rounded to fp16 (never raw random bits, which could be NaN or Inf);
every other byte is drawn uniformly, except where a distribution below says otherwise.
Field offsets follow the public GGUF block definitions:

  Q8_0   34 B: fp16 d @0, int8 q[32] @2            d ~ U[1e-3,2e-3], q ~ U{-127..127}
  Q4_0   18 B: fp16 d @0, nibbles @2                d ~ U[1e-3,2e-3], nibble bytes uniform
  Q4_1   20 B: fp16 d @0, fp16 m @2, nibbles @4     d as Q4_0, m ~ U[-1e-3,1e-3]
  Q5_0   22 B: fp16 d @0, qh @2, nibbles @6         d as Q4_0, qh and nibble bytes uniform
  Q5_1   24 B: fp16 d @0, fp16 m @2, qh @4, nib @8  d, m as Q4_1
  IQ4_NL 18 B: fp16 d @0, indices @2                d as Q4_0, index bytes uniform
  Q4_K  144 B: fp16 d @0, fp16 dmin @2, rest bytes  d ~ U[1e-3,2e-3], dmin ~ U[0,1e-3]
  Q5_K  176 B: as Q4_K (the qh bytes are uniform too)
  Q6_K  210 B: ql/qh @0..191 uniform, int8 sc[16] @192 ~ U{-127..127}, fp16 d @208
  Q2_K   84 B: scale|min bytes @0..15 and codes @16..79 uniform, fp16 d @80, fp16 dmin @82
               (d, dmin as Q4_K)
  Q3_K  110 B: hmask, codes and packed scales @0..107 uniform, fp16 d @108 ~ U[1e-3,2e-3]
  IQ4_XS 136 B: fp16 d @0, scales and indices uniform bytes
"""
from __future__ import annotations

import numpy as np

Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K, IQ4_NL, IQ4_XS = 2, 3, 6, 7, 8, 12, 13, 14, 20, 23
Q2_K, Q3_K = 10, 11
FORMATS = {"Q4_0": Q4_0, "Q4_1": Q4_1, "Q5_0": Q5_0, "Q5_1": Q5_1, "Q8_0": Q8_0, "Q2_K": Q2_K, "Q3_K": Q3_K,
           "Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K, "IQ4_NL": IQ4_NL, "IQ4_XS": IQ4_XS}
FORMAT_NAMES = {v: k for k, v in FORMATS.items()}
BLOCK_ELEMS = {Q4_0: 32, Q4_1: 32, Q5_0: 32, Q5_1: 32, Q8_0: 32, Q2_K: 256, Q3_K: 256, Q4_K: 256, Q5_K: 256,
               Q6_K: 256, IQ4_NL: 32, IQ4_XS: 256}
BLOCK_BYTES = {Q4_0: 18, Q4_1: 20, Q5_0: 22, Q5_1: 24, Q8_0: 34, Q2_K: 84, Q3_K: 110, Q4_K: 144, Q5_K: 176,
               Q6_K: 210, IQ4_NL: 18, IQ4_XS: 136}

BASE_SEED = 0x51472026


def seed_for(config_id: int, salt: int = 0) -> int:
    """Seed of workload ``config_id`` (1..5); ``salt`` separates independent tensors."""
    return BASE_SEED + int(config_id) + 1000003 * int(salt)


def rng(config_id: int, salt: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed_for(config_id, salt))


def row_bytes(fmt: int, K: int) -> int:
    return (K // BLOCK_ELEMS[fmt]) * BLOCK_BYTES[fmt]


def matrix_bytes(fmt: int, N: int, K: int) -> int:
    return N * row_bytes(fmt, K)


def _put_half(blocks: np.ndarray, off: int, values: np.ndarray) -> None:
    h = values.astype(np.float16).view(np.uint8).reshape(-1, 2)
    blocks[:, off:off + 2] = h


def weights(fmt: int, N: int, K: int, g: np.random.Generator) -> np.ndarray:
    """N x K matrix of ``fmt`` blocks, rows contiguous: uint8 array (N, row_bytes)."""
    qk, bs = BLOCK_ELEMS[fmt], BLOCK_BYTES[fmt]
    if K % qk:
        raise ValueError(f"K={K} is not a multiple of the block size {qk}")
    nblk = N * (K // qk)
    blocks = g.integers(0, 256, size=(nblk, bs), dtype=np.uint8)
    d = g.uniform(1e-3, 2e-3, size=nblk).astype(np.float32)
    if fmt == Q8_0:
        _put_half(blocks, 0, d)
        blocks[:, 2:34] = g.integers(-127, 128, size=(nblk, 32), dtype=np.int16).astype(np.int8).view(np.uint8)
    elif fmt in (Q4_0, IQ4_XS, IQ4_NL, Q5_0):
        _put_half(blocks, 0, d)
    elif fmt in (Q4_1, Q5_1):
        _put_half(blocks, 0, d)
        _put_half(blocks, 2, g.uniform(-1e-3, 1e-3, size=nblk).astype(np.float32))
    elif fmt in (Q4_K, Q5_K):
        _put_half(blocks, 0, d)
        _put_half(blocks, 2, g.uniform(0.0, 1e-3, size=nblk).astype(np.float32))
    elif fmt == Q2_K:
        _put_half(blocks, 80, d)
        _put_half(blocks, 82, g.uniform(0.0, 1e-3, size=nblk).astype(np.float32))
    elif fmt == Q3_K:
        _put_half(blocks, 108, d)
    elif fmt == Q6_K:
        blocks[:, 192:208] = g.integers(-127, 128, size=(nblk, 16), dtype=np.int16).astype(np.int8).view(np.uint8)
        _put_half(blocks, 208, d)
    else:
        raise ValueError(f"unknown format {fmt}")
    return blocks.reshape(N, (K // qk) * bs)


def activations(M: int, K: int, g: np.random.Generator) -> np.ndarray:
    """x ~ N(0, 1), fp32, M x K."""
    return g.standard_normal(size=(M, K), dtype=np.float32)


def router_weights(E: int, H: int, g: np.random.Generator) -> np.ndarray:
    """Router matrix E x H, fp32 ~ N(0, 1/H) so that logits of N(0,1) inputs are ~N(0,1)."""
    return (g.standard_normal(size=(E, H), dtype=np.float32) / np.float32(np.sqrt(H))).astype(np.float32)


def stacked_experts(fmt: int, E: int, N: int, K: int, g: np.random.Generator) -> np.ndarray:
    """E matrices of N x K stacked contiguously: uint8 (E, N, row_bytes)."""
    return weights(fmt, E * N, K, g).reshape(E, N, row_bytes(fmt, K))
