// qg_dequant.cuh -- fp16 dequantization of one 32-element unit of a GGUF row, for the
// prefill GEMM on tensor cores.
//
// "01 · 阶段总览：从 2B 到 8B 再到 MoE", section 九: prefill moved to the tensor cores with
// the weights dequantized to fp16 inside the kernel (a fused fp16 path).  The operand is
// formed per unit u of 32 elements as
//     w32 = A_u * c_e - B_u * mc_e     (fp32; both products exact, one rounding)
//     w16 = round-to-nearest-even fp16 of w32
// with, per format (public GGUF block layouts; offsets in bytes):
//   Q4_0, IQ4_NL  18 B  d@0, qs@2          A = d, c = nib - 8 (Q4_0), codebook[nib] (IQ4_NL)
//   Q4_1          20 B  d@0, m@2, qs@4     A = d, c = nib, B*mc = -m
//   Q5_0          22 B  d@0, qh@2, qs@6    A = d, c = (nib | bit e of qh << 4) - 16
//   Q5_1          24 B  d@0, m@2, qh@4, qs@8   A = d, c = nib | bit << 4, B*mc = -m
//   Q8_0          34 B  d@0, q@2           A = d, c = q
//   Q2_K          84 B  sc@0, qs@16, d@80, dmin@82   e = 128h+32j+l: q = qs[32h+l] >> 2j & 3,
//                                          A = d, c = (sc[e/16] & 15) * q, B = dmin, mc = sc[e/16] >> 4
//   Q3_K         110 B  hmask@0, qs@32, sc12@96, d@108   c = (scale6(e/16) - 32) *
//                                          (q - 4 * !(hmask[l] >> (4h+j) & 1)), A = d
//   Q4_K         144 B  d@0, dmin@2, sc12@4, qs@16   unit j: A = d*S_j, B = dmin*M_j, c = nibble
//   Q5_K         176 B  as Q4_K, qh@16, qs@48         c += 16 * (qh[l] >> j & 1)
//   Q6_K         210 B  ql@0, qh@128, sc@192, d@208  c = sc[e/16] * (q6 - 32), A = d
//   IQ4_XS       136 B  d@0, scales_h@2, scales_l@4, qs@8   A = d*(ls-32), c = codebook[idx]
// Every weight is read with loads of its natural alignment (2, 4, 8 or 16 bytes), never past
// its block, so a unit is fetched without touching bytes outside the tensor.
//
// fetch() loads the words one unit needs (so that a kernel can issue the loads of later units
// before it converts the current one); convert() forms the 32 fp16 values, packed two per
// 32-bit word in element order (the lower element in the low half).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "qg_common.cuh"

namespace qg {

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p));
}
__device__ __forceinline__ uint32_t ldg_u32(const uint8_t *p) { return __ldg(reinterpret_cast<const unsigned int *>(p)); }
__device__ __forceinline__ uint4 ldg_u128(const uint8_t *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
// a 32-bit word at a 2-byte-aligned address
__device__ __forceinline__ uint32_t ldg_w2(const uint8_t *p) { return ldg_u16(p) | (ldg_u16(p + 2) << 16); }

__device__ __forceinline__ uint32_t byte_at(uint32_t w, int k) { return (w >> (8 * k)) & 255u; }
// Byte b of a word array; b may be a run-time value (a select chain keeps w in registers).
template <int NW>
__device__ __forceinline__ uint32_t byte_of_words(const uint32_t (&w)[NW], int b) {
    uint32_t word = w[0];
#pragma unroll
    for (int i = 1; i < NW; ++i)
        if ((b >> 2) == i) word = w[i];
    return byte_at(word, b & 3);
}
__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// The 16-entry IQ4_NL codebook, four entries per word, selected with byte permutes.
constexpr uint32_t cb4(int i) {
    constexpr int8_t t[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};
    return (uint32_t)(uint8_t)t[i] | ((uint32_t)(uint8_t)t[i + 1] << 8) | ((uint32_t)(uint8_t)t[i + 2] << 16) |
           ((uint32_t)(uint8_t)t[i + 3] << 24);
}
__device__ __forceinline__ int codebook(uint32_t idx) {
    const uint32_t lo = prmt(cb4(0), cb4(4), idx & 7u), hi = prmt(cb4(8), cb4(12), idx & 7u);
    return (int)(int8_t)((idx & 8u) ? hi : lo);
}

// Packs fp32 values v[0..31] into 16 words of two fp16 (round to nearest even).
__device__ __forceinline__ void pack_f16(const float (&v)[32], uint32_t (&h)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const __half2 p = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t *>(&p);
    }
}

// Q4_K / Q5_K: 6-bit scale and min of sub-block j from the 12 packed bytes sc (bytes 4..15 of
// the block, i.e. bytes 0..11 of the 16-byte header words h[1..3]).
__device__ __forceinline__ void kq_scale_min(const uint32_t (&hdr)[4], int j, int &S, int &M) {
    auto sc = [&](int b) { return (int)byte_of_words(hdr, 4 + b); };
    if (j < 4) {
        S = sc(j) & 63;
        M = sc(j + 4) & 63;
    } else {
        S = (sc(j + 4) & 15) | ((sc(j - 4) >> 6) << 4);
        M = (sc(j + 4) >> 4) | ((sc(j) >> 6) << 4);
    }
}

template <int FMT>
struct Deq;

// ---------------------------------------------------------------- 32-element blocks
template <int FMT>
struct DeqLegacy {
    static constexpr int BS = FMT == F_Q8_0 ? 34 : FMT == F_Q4_1 ? 20 : FMT == F_Q5_0 ? 22 : FMT == F_Q5_1 ? 24 : 18;
    static constexpr int QK = 32;
    static constexpr bool HAS_M = FMT == F_Q4_1 || FMT == F_Q5_1;
    static constexpr bool HAS_QH = FMT == F_Q5_0 || FMT == F_Q5_1;
    static constexpr int NQ = FMT == F_Q8_0 ? 8 : 4;  // code words
    static constexpr int RW = 2 + NQ;                 // w[0] d (| m << 16), w[1] qh, w[2..] codes
    using Raw = uint32_t[RW];

    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, Raw &r) {
        const uint8_t *b = row + (size_t)u * BS;
        if constexpr (FMT == F_Q4_1 || FMT == F_Q5_1) {  // 4- and 8-byte-aligned blocks
            r[0] = ldg_u32(b);
            r[1] = FMT == F_Q5_1 ? ldg_u32(b + 4) : 0u;
            const int qs = FMT == F_Q5_1 ? 8 : 4;
#pragma unroll
            for (int i = 0; i < NQ; ++i) r[2 + i] = ldg_u32(b + qs + 4 * i);
        } else {  // 2-byte-aligned blocks
            r[0] = ldg_u16(b);
            r[1] = FMT == F_Q5_0 ? ldg_w2(b + 2) : 0u;
            const int qs = FMT == F_Q5_0 ? 6 : 2;
#pragma unroll
            for (int i = 0; i < NQ; ++i) r[2 + i] = ldg_w2(b + qs + 4 * i);
        }
    }

    __device__ __forceinline__ static void convert(const Raw &r, uint32_t (&h)[16]) {
        const float d = half_lo(r[0]);
        const float m = HAS_M ? half_hi(r[0]) : 0.0f;
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            int c;
            if constexpr (FMT == F_Q8_0) {
                c = (int)(int8_t)byte_at(r[2 + e / 4], e % 4);
            } else {
                const int k = e % 16;
                const uint32_t byte = byte_at(r[2 + k / 4], k % 4);
                c = (int)(e < 16 ? (byte & 15u) : (byte >> 4));
                if constexpr (HAS_QH) c |= (int)((r[1] >> e) & 1u) << 4;
                if constexpr (FMT == F_Q4_0) c -= 8;
                if constexpr (FMT == F_Q5_0) c -= 16;
                if constexpr (FMT == F_IQ4_NL) c = codebook((uint32_t)c);
            }
            // d * c is exact in fp32; with the additive min one rounding: RN(d*c + m)
            v[e] = HAS_M ? fmaf(d, (float)c, m) : d * (float)c;
        }
        pack_f16(v, h);
    }
};
template <> struct Deq<F_Q4_0> : DeqLegacy<F_Q4_0> {};
template <> struct Deq<F_Q4_1> : DeqLegacy<F_Q4_1> {};
template <> struct Deq<F_Q5_0> : DeqLegacy<F_Q5_0> {};
template <> struct Deq<F_Q5_1> : DeqLegacy<F_Q5_1> {};
template <> struct Deq<F_Q8_0> : DeqLegacy<F_Q8_0> {};
template <> struct Deq<F_IQ4_NL> : DeqLegacy<F_IQ4_NL> {};

// ---------------------------------------------------------------- 256-element superblocks
template <>
struct Deq<F_Q2_K> {
    static constexpr int BS = 84, QK = 256, RW = 10;  // sc pair, d|dmin, 8 code words
    using Raw = uint32_t[RW];
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, Raw &r) {
        const uint8_t *b = row + (size_t)(u / 8) * BS;
        const int v = u % 8, hh = v / 4;
        r[0] = ldg_u16(b + 2 * v);   // scale|min bytes of sub-blocks 2v, 2v + 1
        r[1] = ldg_u32(b + 80);      // d, dmin
#pragma unroll
        for (int i = 0; i < 8; ++i) r[2 + i] = ldg_u32(b + 16 + 32 * hh + 4 * i);
    }
    __device__ __forceinline__ static void convert_u(const Raw &r, int u, uint32_t (&h)[16]) {
        const int j = (u % 8) % 4;
        const float d = half_lo(r[1]), dmin = half_hi(r[1]);
        float v[32];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const uint32_t sm = byte_at(r[0], l / 16);
            const int q = (int)((byte_at(r[2 + l / 4], l % 4) >> (2 * j)) & 3u);
            const float bm = dmin * (float)(sm >> 4);      // exact
            v[l] = fmaf(d, (float)((int)(sm & 15u) * q), -bm);
        }
        pack_f16(v, h);
    }
};

template <>
struct Deq<F_Q3_K> {
    static constexpr int BS = 110, QK = 256, RW = 18;  // 8 hmask, 8 code words, scale bytes, d
    using Raw = uint32_t[RW];
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, Raw &r) {
        const uint8_t *b = row + (size_t)(u / 8) * BS;
        const int v = u % 8, hh = v / 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = ldg_w2(b + 4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) r[8 + i] = ldg_w2(b + 32 + 32 * hh + 4 * i);
        // sub-blocks 2v, 2v + 1: low nibbles in bytes (2v) % 8, +1; high pairs in 8 + (2v) % 4, +1
        r[16] = ldg_u16(b + 96 + (2 * v) % 8) | (ldg_u16(b + 96 + 8 + (2 * v) % 4) << 16);
        r[17] = ldg_u16(b + 108);
    }
    __device__ __forceinline__ static void convert_u(const Raw &r, int u, uint32_t (&h)[16]) {
        const int v = u % 8, hh = v / 4, j = v % 4;
        const float d = half_lo(r[17]);
        int scale[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int i = 2 * v + s;
            const int low4 = (int)(i < 8 ? (byte_at(r[16], s) & 15u) : (byte_at(r[16], s) >> 4));
            const int high2 = (int)((byte_at(r[16], 2 + s) >> (2 * (i / 4))) & 3u);
            scale[s] = (low4 | (high2 << 4)) - 32;
        }
        float vv[32];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const int q = (int)((byte_at(r[8 + l / 4], l % 4) >> (2 * j)) & 3u);
            const int hb = (int)((byte_at(r[l / 4], l % 4) >> (4 * hh + j)) & 1u);
            vv[l] = d * (float)(scale[l / 16] * (q - (hb ? 0 : 4)));
        }
        pack_f16(vv, h);
    }
};

template <int FMT>
struct DeqKQ {  // Q4_K, Q5_K
    static constexpr bool Q5 = FMT == F_Q5_K;
    static constexpr int BS = Q5 ? 176 : 144, QK = 256, RW = Q5 ? 20 : 12;
    using Raw = uint32_t[RW];  // header (d, dmin, sc12), [qh 32 B], qs 32 B
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, Raw &r) {
        const uint8_t *b = row + (size_t)(u / 8) * BS;
        const int j = u % 8;
        auto put = [&](int at, uint4 x) { r[at] = x.x; r[at + 1] = x.y; r[at + 2] = x.z; r[at + 3] = x.w; };
        put(0, ldg_u128(b));
        const uint8_t *qs = b + (Q5 ? 48 : 16) + 32 * (j / 2);
        put(4, ldg_u128(qs));
        put(8, ldg_u128(qs + 16));
        if constexpr (Q5) {
            put(12, ldg_u128(b + 16));
            put(16, ldg_u128(b + 32));
        }
    }
    __device__ __forceinline__ static void convert_u(const Raw &r, int u, uint32_t (&h)[16]) {
        const int j = u % 8;
        uint32_t hdr[4] = {r[0], r[1], r[2], r[3]};
        int S, M;
        kq_scale_min(hdr, j, S, M);
        const float A = half_lo(r[0]) * (float)S, Bm = half_hi(r[0]) * (float)M;  // exact
        float v[32];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const uint32_t byte = byte_at(r[4 + l / 4], l % 4);
            int c = (int)((j & 1) ? (byte >> 4) : (byte & 15u));
            if constexpr (Q5) c += 16 * (int)((byte_at(r[12 + l / 4], l % 4) >> j) & 1u);
            v[l] = fmaf(A, (float)c, -Bm);
        }
        pack_f16(v, h);
    }
};
template <> struct Deq<F_Q4_K> : DeqKQ<F_Q4_K> {};
template <> struct Deq<F_Q5_K> : DeqKQ<F_Q5_K> {};

template <>
struct Deq<F_Q6_K> {
    static constexpr int BS = 210, QK = 256, RW = 18;  // 8 ql words, 8 qh words, sc pair, d
    using Raw = uint32_t[RW];
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, Raw &r) {
        const uint8_t *b = row + (size_t)(u / 8) * BS;
        const int v = u % 8, hh = v / 4, t = v % 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = ldg_w2(b + 64 * hh + 32 * (t & 1) + 4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) r[8 + i] = ldg_w2(b + 128 + 32 * hh + 4 * i);
        r[16] = ldg_u16(b + 192 + 2 * v);  // int8 sub-scales of elements 0..15 and 16..31
        r[17] = ldg_u16(b + 208);
    }
    __device__ __forceinline__ static void convert_u(const Raw &r, int u, uint32_t (&h)[16]) {
        const int t = (u % 8) % 4;
        const float d = half_lo(r[17]);
        float v[32];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const uint32_t lb = byte_at(r[l / 4], l % 4);
            const int low4 = (int)(t < 2 ? (lb & 15u) : (lb >> 4));
            const int hi2 = (int)((byte_at(r[8 + l / 4], l % 4) >> (2 * t)) & 3u);
            const int sc = (int)(int8_t)byte_at(r[16], l / 16);
            v[l] = d * (float)(sc * ((low4 | (hi2 << 4)) - 32));  // exact
        }
        pack_f16(v, h);
    }
};

template <>
struct Deq<F_IQ4_XS> {
    static constexpr int BS = 136, QK = 256, RW = 6;  // d | scales_h, scales_l, 4 index words
    using Raw = uint32_t[RW];
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, Raw &r) {
        const uint8_t *b = row + (size_t)(u / 8) * BS;
        const int ib = u % 8;
        r[0] = ldg_u32(b);
        r[1] = ldg_u32(b + 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) r[2 + i] = ldg_u32(b + 8 + 16 * ib + 4 * i);
    }
    __device__ __forceinline__ static void convert_u(const Raw &r, int u, uint32_t (&h)[16]) {
        const int ib = u % 8;
        const int ls = (int)((byte_at(r[1], ib / 2) >> (4 * (ib % 2))) & 15u) | (int)(((r[0] >> (16 + 2 * ib)) & 3u) << 4);
        const float A = half_lo(r[0]) * (float)(ls - 32);  // exact
        float v[32];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const int k = l % 16;
            const uint32_t byte = byte_at(r[2 + k / 4], k % 4);
            v[l] = A * (float)codebook(l < 16 ? (byte & 15u) : (byte >> 4));
        }
        pack_f16(v, h);
    }
};

// Uniform entry: the unit index matters to the superblock formats' convert.
template <int FMT>
__device__ __forceinline__ void deq_convert(const typename Deq<FMT>::Raw &r, int u, uint32_t (&h)[16]) {
    if constexpr (Deq<FMT>::QK == 32)
        Deq<FMT>::convert(r, h);
    else
        Deq<FMT>::convert_u(r, u, h);
}

}  // namespace qg
