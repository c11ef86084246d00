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

// The NW words at byte address p (2-byte aligned, p + 2 * NB16 the end of the bytes that are
// needed: NB16 16-bit units) read through the aligned 16-byte chunks that cover them, when
// those chunks lie below lim (the end of the tensor), and realigned in registers: shifts by
// 8, 4 and 2 bytes of the offset within the first chunk (MAXO: the largest such offset the
// caller can have).  Otherwise (a window reaching past the tensor's end) the needed 16-bit
// units are loaded one by one and the rest of the words are zero.
template <int NW, int NB16, int MAXO>
__device__ __forceinline__ void fetch_words(const uint8_t *p, const uint8_t *lim, uint32_t (&out)[NW]) {
    constexpr int NC = (MAXO + 2 * NB16 + 15) / 16;  // chunks covering the needed bytes at the worst offset
    const uint8_t *base = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)15);
    const uint32_t o = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 15u);
    if (base + 16 * NC <= lim) {
        uint32_t w[4 * NC + 3];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 v = ldg_u128(base + 16 * c);
            w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
        w[4 * NC] = w[4 * NC + 1] = w[4 * NC + 2] = 0u;
#pragma unroll
        for (int i = 0; i < 4 * NC + 1; ++i) w[i] = (o & 8u) ? w[i + 2] : w[i];
#pragma unroll
        for (int i = 0; i < 4 * NC; ++i) w[i] = (o & 4u) ? w[i + 1] : w[i];
#pragma unroll
        for (int i = 0; i < NW; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], 8u * (o & 2u));
    } else {
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint32_t lo = 2 * i < NB16 ? ldg_u16(p + 4 * i) : 0u;
            const uint32_t hi = 2 * i + 1 < NB16 ? ldg_u16(p + 4 * i + 2) : 0u;
            out[i] = lo | (hi << 16);
        }
    }
}

// Packs fp32 values v[0..31] into 16 words of two fp16 (round to nearest even).
__device__ __forceinline__ void pack_f16(const float (&v)[32], uint32_t (&h)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const __half2 p = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t *>(&p);
    }
}

// Byte k (k = 0..3) of w as the fp32 value 2^23 + byte: the byte becomes the low mantissa
// bits of 2^23 (exponent byte 0x4B), so subtracting 2^23 (+ an offset) afterwards is exact.
constexpr float MAGIC = 8388608.0f;  // 2^23
__device__ __forceinline__ float byte_magic(uint32_t w, int k) {
    return __uint_as_float(prmt(w, 0x4B000000u, 0x7440u + (uint32_t)k));
}
// Four small unsigned integers held in the bytes of w, minus off, as exact fp32 values.
__device__ __forceinline__ void bytes4_to_f32(uint32_t w, float off, float *f) {
#pragma unroll
    for (int k = 0; k < 4; ++k) f[k] = byte_magic(w, k) - (MAGIC + off);
}

// The codebook values of the 8 indices in q (byte b: low nibble = element b of the unit's
// first half, high nibble = element b of its second half), each plus 128: lo holds elements
// 0..3 of the first half, hi elements 0..3 of the second half, one per byte.
__device__ __forceinline__ void codebook8_biased(uint32_t q, uint32_t &lo, uint32_t &hi) {
    const uint32_t i7 = q & 0x77777777u;
    const uint32_t pick = ((q >> 1) & 0x44444444u) | 0x32103210u;
    const uint32_t a0 = prmt(cb4(0), cb4(4), i7), b0 = prmt(cb4(8), cb4(12), i7);
    const uint32_t a1 = prmt(cb4(0), cb4(4), i7 >> 16), b1 = prmt(cb4(8), cb4(12), i7 >> 16);
    const uint32_t A = prmt(a0, b0, pick), B = prmt(a1, b1, pick >> 16);
    lo = prmt(A, B, 0x6420u) ^ 0x80808080u;
    hi = prmt(A, B, 0x7531u) ^ 0x80808080u;
}

// Q4_K / Q5_K: 6-bit scale S and min M of sub-block j (0..7) from the 12 packed scale bytes
// sc[0..11] = the header words h1 (sc 0..3), h2 (sc 4..7), h3 (sc 8..11):
//   j < 4:  S = sc[j] & 63,                          M = sc[j+4] & 63
//   j >= 4: S = (sc[j+4] & 15) | (sc[j-4] >> 6) << 4,  M = (sc[j+4] >> 4) | (sc[j] >> 6) << 4
// (run-time shifts of the words; no array indexing).
__device__ __forceinline__ void kq_scale_min(uint32_t h1, uint32_t h2, uint32_t h3, int j, int &S, int &M) {
    const int e = 8 * (j & 3);
    if (j < 4) {
        S = (int)((h1 >> e) & 63u);
        M = (int)((h2 >> e) & 63u);
    } else {
        S = (int)(((h3 >> e) & 15u) | (((h1 >> (e + 6)) & 3u) << 4));
        M = (int)(((h3 >> (e + 4)) & 15u) | (((h2 >> (e + 6)) & 3u) << 4));
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

    // the block's words through aligned 16-byte loads of its window (fetch_words), then the
    // fields: w[0] = d (| m << 16), w[1] = qh, w[2..] = code words
    static constexpr int NWB = FMT == F_Q8_0 ? 9 : (FMT == F_Q5_0 || FMT == F_Q5_1) ? 6 : 5;  // words used
    static constexpr int MAXO = FMT == F_Q5_1 ? 8 : FMT == F_Q4_1 ? 12 : 14;
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, const uint8_t *lim, Raw &r) {
        const uint8_t *b = row + (size_t)u * BS;
        uint32_t w[NWB];
        fetch_words<NWB, BS / 2, MAXO>(b, lim, w);
        if constexpr (FMT == F_Q4_1 || FMT == F_Q5_1) {  // 4-byte-aligned fields
            r[0] = w[0];
            r[1] = FMT == F_Q5_1 ? w[1] : 0u;
            const int qs = FMT == F_Q5_1 ? 2 : 1;
#pragma unroll
            for (int i = 0; i < NQ; ++i) r[2 + i] = w[qs + i];
        } else {  // fields after the 2-byte d: realigned by 16 bits
            r[0] = w[0] & 0xffffu;
            r[1] = FMT == F_Q5_0 ? __funnelshift_r(w[0], w[1], 16) : 0u;
            const int qs = FMT == F_Q5_0 ? 1 : 0;  // word holding the code bytes' first half
#pragma unroll
            for (int i = 0; i < NQ; ++i) r[2 + i] = __funnelshift_r(w[qs + i], w[qs + i + 1], 16);
        }
    }

    __device__ __forceinline__ static void convert(const Raw &r, uint32_t (&h)[16]) {
        const float d = half_lo(r[0]);
        const float m = HAS_M ? half_hi(r[0]) : 0.0f;
        float v[32];
        // element codes four per word, then exact fp32 values: d * c (one exact product), or
        // RN(d * c + m) for the additive-min formats
        auto emit = [&](int e0, uint32_t w, float off) {
            float f[4];
            bytes4_to_f32(w, off, f);
#pragma unroll
            for (int k = 0; k < 4; ++k) v[e0 + k] = HAS_M ? fmaf(d, f[k], m) : d * f[k];
        };
        if constexpr (FMT == F_Q8_0) {
#pragma unroll
            for (int k = 0; k < 8; ++k) emit(4 * k, r[2 + k] ^ 0x80808080u, 128.0f);  // int8 + 128
        } else if constexpr (FMT == F_IQ4_NL) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t lo, hi;  // codebook values + 128 of elements 4k.. and 16 + 4k..
                codebook8_biased(r[2 + k], lo, hi);
                emit(4 * k, lo, 128.0f);
                emit(16 + 4 * k, hi, 128.0f);
            }
        } else {
            constexpr float OFF = FMT == F_Q4_0 ? 8.0f : FMT == F_Q5_0 ? 16.0f : 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t lo = r[2 + k] & 0x0f0f0f0fu, hi = (r[2 + k] >> 4) & 0x0f0f0f0fu;
                if constexpr (HAS_QH) {  // the fifth bits of elements 4k.. and 16 + 4k..
                    lo |= ((((r[1] >> (4 * k)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
                    hi |= ((((r[1] >> (16 + 4 * k)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
                }
                emit(4 * k, lo, OFF);
                emit(16 + 4 * k, hi, OFF);
            }
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
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, const uint8_t *, Raw &r) {
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
        for (int hh = 0; hh < 2; ++hh) {  // 16-element sub-blocks of the unit
            const uint32_t sm = byte_at(r[0], hh);
            const float dS = d * (float)(sm & 15u), bm = dmin * (float)(sm >> 4);  // exact
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float f[4];
                bytes4_to_f32((r[2 + 4 * hh + k] >> (2 * j)) & 0x03030303u, 0.0f, f);
                // RN(d * (S q) - dmin * M): the product d S q is exact
#pragma unroll
                for (int i = 0; i < 4; ++i) v[16 * hh + 4 * k + i] = fmaf(dS, f[i], -bm);
            }
        }
        pack_f16(v, h);
    }
};

template <>
struct Deq<F_Q3_K> {
    static constexpr int BS = 110, QK = 256, RW = 18;  // 8 hmask, 8 code words, scale bytes, d
    using Raw = uint32_t[RW];
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, const uint8_t *, Raw &r) {
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
        float vv[32];
#pragma unroll
        for (int s = 0; s < 2; ++s) {  // 16-element sub-blocks 2v + s
            const int i = 2 * v + s;
            const int low4 = (int)(i < 8 ? (byte_at(r[16], s) & 15u) : (byte_at(r[16], s) >> 4));
            const int high2 = (int)((byte_at(r[16], 2 + s) >> (2 * (i / 4))) & 3u);
            const float sc = (float)((low4 | (high2 << 4)) - 32);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // code byte q | hb << 2 in 0..7; the value is q - 4 * (1 - hb) = byte - 4
                const uint32_t q = (r[8 + 4 * s + k] >> (2 * j)) & 0x03030303u;
                const uint32_t hb = (r[4 * s + k] >> (4 * hh + j)) & 0x01010101u;
                float f[4];
                bytes4_to_f32(q | (hb << 2), 4.0f, f);
                // the integer code c = scale * (byte - 4) (adding +0 makes a zero +0, as the
                // integer product is), then d * c
#pragma unroll
                for (int e = 0; e < 4; ++e) vv[16 * s + 4 * k + e] = d * fmaf(sc, f[e], 0.0f);
            }
        }
        pack_f16(vv, h);
    }
};

template <int FMT>
struct DeqKQ {  // Q4_K, Q5_K
    static constexpr bool Q5 = FMT == F_Q5_K;
    static constexpr int BS = Q5 ? 176 : 144, QK = 256, RW = Q5 ? 20 : 12;
    using Raw = uint32_t[RW];  // header (d, dmin, sc12), [qh 32 B], qs 32 B
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, const uint8_t *, Raw &r) {
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
        int S, M;
        kq_scale_min(r[1], r[2], r[3], j, S, M);
        const float A = half_lo(r[0]) * (float)S, Bm = half_hi(r[0]) * (float)M;  // exact
        const int sh = 4 * (j & 1);
        float v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            uint32_t c = (r[4 + k] >> sh) & 0x0f0f0f0fu;
            if constexpr (Q5) c |= ((r[12 + k] >> j) & 0x01010101u) << 4;
            float f[4];
            bytes4_to_f32(c, 0.0f, f);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[4 * k + i] = fmaf(A, f[i], -Bm);
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
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, const uint8_t *, Raw &r) {
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
        for (int hh = 0; hh < 2; ++hh) {  // 16-element sub-blocks: their int8 scales
            const float sc = (float)(int)(int8_t)byte_at(r[16], hh);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lw = r[4 * hh + k], qw = r[8 + 4 * hh + k];
                const uint32_t q6 = ((t < 2 ? lw : (lw >> 4)) & 0x0f0f0f0fu) | (((qw >> (2 * t)) & 0x03030303u) << 4);
                float f[4];
                bytes4_to_f32(q6, 32.0f, f);
                // the integer code c = sc * (q6 - 32) (a zero made +0, as the integer product
                // is), then d * c: both products exact
#pragma unroll
                for (int i = 0; i < 4; ++i) v[16 * hh + 4 * k + i] = d * fmaf(sc, f[i], 0.0f);
            }
        }
        pack_f16(v, h);
    }
};

template <>
struct Deq<F_IQ4_XS> {
    static constexpr int BS = 136, QK = 256, RW = 6;  // d | scales_h, scales_l, 4 index words
    using Raw = uint32_t[RW];
    __device__ __forceinline__ static void fetch(const uint8_t *row, int u, const uint8_t *, Raw &r) {
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
        for (int k = 0; k < 4; ++k) {
            uint32_t lo, hi;
            codebook8_biased(r[2 + k], lo, hi);
            float f[4];
            bytes4_to_f32(lo, 128.0f, f);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[4 * k + i] = A * f[i];
            bytes4_to_f32(hi, 128.0f, f);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[16 + 4 * k + i] = A * f[i];
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
