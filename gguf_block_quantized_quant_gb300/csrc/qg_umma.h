// qg_umma.h -- encodings of the 5th-generation tensor-core (tcgen05) descriptors used by the
// prefill GEMM, as plain host/device functions so that a CPU test can check every field.
//
// Shared-memory matrix descriptor (64 bits):
//   bits  0-13  start address >> 4 (shared-window address, 18 bits significant)
//   bits 16-29  leading-dimension byte offset >> 4 (unused for swizzled K-major operands)
//   bits 32-45  stride-dimension byte offset >> 4 (distance between 8-row groups)
//   bits 46-48  fixed value 0b001
//   bits 49-51  matrix base offset (0: every swizzle atom starts 1024-byte aligned)
//   bit  52     leading-dimension stride mode (0: relative)
//   bits 61-63  swizzle: 0 none, 1 128-byte with 32-byte atoms, 2 128-byte, 4 64-byte, 6 32-byte
// Instruction descriptor of kind::f16 (32 bits):
//   bits 0-1 sparsity selector, 2 sparsity, 3 saturate (all 0 here)
//   bits 4-5 D type (1 = fp32)     bits 7-9 A type (0 = fp16, 1 = bf16)   bits 10-12 B type
//   bit 13/14 negate A/B           bit 15/16 A/B major (0 = K-major)
//   bits 17-22 N >> 3              bit 23 reserved
//   bits 24-28 M >> 4              bit 29 reserved             bits 30-31 max shift (0)
// Operand layout (K-major, 128-byte swizzle): an operand tile of R rows and 64 fp16 of K is R
// rows of 128 bytes; rows r..r+7 (r a multiple of 8) form a 1024-byte atom, atoms are
// packed (stride-dimension offset 1024); inside an atom the 16-byte chunk c of row r sits at
// chunk position c ^ (r & 7).  An MMA step of K = 16 (32 bytes) at chunk pair 2k, 2k + 1 is
// addressed by advancing the start address by 32 k bytes.
#pragma once

#include <stdint.h>

namespace qg {

constexpr uint32_t UMMA_SW128 = 2;      // swizzle mode field: 128-byte swizzle
constexpr uint32_t UMMA_ATOM_BYTES = 1024;

__host__ __device__ constexpr uint64_t umma_smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                                      uint32_t swizzle) {
    return (uint64_t)((smem_addr & 0x3ffffu) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo_bytes >> 4) & 0x3fffu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)(swizzle & 7u) << 61);
}

// The descriptor of a K-major, 128-byte-swizzled fp16 tile at smem_addr (1024-byte aligned).
__host__ __device__ constexpr uint64_t umma_desc_kmajor_sw128(uint32_t smem_addr) {
    return umma_smem_desc(smem_addr, 16, UMMA_ATOM_BYTES, UMMA_SW128);
}

// kind::f16 instruction descriptor: fp16 A and B (both K-major), fp32 accumulator, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of fp16 element (row r, k) inside a K-major 128-byte-swizzled tile of 64 k.
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t r, uint32_t k) {
    return r * 128u + ((((k >> 3) ^ (r & 7u)) & 7u) << 4) + (k & 7u) * 2u;
}

// Shapes the prefill GEMM issues: M = 128 rows per CTA (cta_group::1); N a multiple of 16 up
// to 256; K = 16 per instruction; TMEM columns: the power of two >= the CTA's accumulator
// columns (up to two accumulators of N), at least 32.
constexpr int PF_BM = 128;
constexpr int PF_BK = 64;
constexpr int PF_MAX_BT = 256;
__host__ __device__ constexpr bool umma_shape_ok(int M, int N) { return M == 128 && N >= 16 && N <= 256 && N % 16 == 0; }
__host__ __device__ constexpr int tmem_cols_for(int n) {
    return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

}  // namespace qg
