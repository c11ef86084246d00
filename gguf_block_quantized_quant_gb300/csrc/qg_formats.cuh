// qg_formats.cuh -- register-resident decoders for the six GGUF block formats.
//
// The GEMV is computed on the raw blocks in place ("为什么专家缓存救不了稠密模型", Q&A
// "如何让CUDA直接计算GGUF混合量化块而不展开为FP16？"): each 32-element unit of a block
// is unpacked in registers into 8 words of four 8-bit codes, dotted with the int8
// activation codes by dp4a, and the fp32 scale factors are applied to the exact int32 sum
// (for K-quants together with the min "correction term"; for IQ4_XS after a register
// lookup in the 16-entry codebook).  Byte layouts are the public GGUF block definitions
// (the pages name the formats but do not print them):
//
//   Q8_0    34 B: fp16 d, int8 q[32]                          w = d*q
//   Q4_0    18 B: fp16 d, qs[16]; e<16 low nibble of qs[e],   w = d*(nib-8)
//                 e>=16 high nibble of qs[e-16]
//   Q4_K   144 B: fp16 d, fp16 dmin, sc12[12], qs[128]        w = d*S_j*code - dmin*M_j
//   Q5_K   176 B: fp16 d, fp16 dmin, sc12[12], qh[32], qs[128] (code += 16*bit j of qh[l])
//   Q6_K   210 B: ql[128], qh[64], int8 sc[16], fp16 d         w = d*sc[e/16]*(code-32)
//   IQ4_XS 136 B: fp16 d, u16 scales_h, scales_l[4], qs[128]  w = d*(ls-32)*K[idx]
//
// All weight reads are from shared memory (32-bit addresses).  Q8_0, Q4_0 and Q6_K blocks
// may start on any even byte, so their fields are fetched as aligned words and realigned
// with byte permutes; Q4_K/Q5_K blocks are 16-byte aligned and IQ4_XS blocks 8-byte aligned
// in every staging layout used here.
#pragma once

#include "qg_common.cuh"

namespace qg {

enum : int { F_Q4_0 = 2, F_Q8_0 = 8, F_Q4_K = 12, F_Q5_K = 13, F_Q6_K = 14, F_IQ4_XS = 23 };

// One decoded 32-element unit.
struct WUnit {
    uint32_t c[8];  // codes, 4 per word, element order (word k holds elements 4k..4k+3)
    float fa;       // main scale of the unit
    float fb;       // min factor (K-quants), else unused
    int sA, sB;     // Q6_K sub-scales of elements 0..15 and 16..31
};

// Activation operand of one unit for one token.
struct XUnit {
    uint32_t q[8];
    float d;
    int s;
};

// Realign 4 bytes starting at byte 2 (sel 0x5432) or byte 4 (sel 0x7654) of {w1:w0}.
__device__ __forceinline__ uint32_t realign(uint32_t w0, uint32_t w1, uint32_t sel) { return prmt(w0, w1, sel); }

template <int FMT>
struct Fmt;

// ------------------------------------------------------------------------------- Q8_0
template <>
struct Fmt<F_Q8_0> {
    static constexpr int QK = 32, BS = 34, UPB = 1;
    static constexpr bool NEED_XS = false;
    __device__ __forceinline__ static void decode(uint32_t blk, int, WUnit &w) {
        const uint32_t a = blk & 3u, base = blk - a;  // a is 0 or 2
        uint32_t wd[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) wd[k] = lds32(base + 4 * k);
        const uint32_t sel = a ? 0x7654u : 0x5432u;
        w.fa = half_bits_to_float(a ? (wd[0] >> 16) : wd[0]);
#pragma unroll
        for (int k = 0; k < 8; ++k) w.c[k] = realign(wd[k], wd[k + 1], sel);
    }
    __device__ __forceinline__ static int idot(const WUnit &w, const XUnit &x) {
        int s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) s = dp4a(w.c[k], x.q[k], s);
        return s;
    }
    __device__ __forceinline__ static float accum(float acc, const WUnit &w, int dot, const XUnit &x) {
        return fmaf(w.fa * x.d, (float)dot, acc);
    }
};

// ------------------------------------------------------------------------------- Q4_0
template <>
struct Fmt<F_Q4_0> {
    static constexpr int QK = 32, BS = 18, UPB = 1;
    static constexpr bool NEED_XS = true;  // the -8 offset is folded in as -8*sum(q)
    __device__ __forceinline__ static void decode(uint32_t blk, int, WUnit &w) {
        const uint32_t a = blk & 3u, base = blk - a;
        uint32_t wd[5];
#pragma unroll
        for (int k = 0; k < 5; ++k) wd[k] = lds32(base + 4 * k);
        const uint32_t sel = a ? 0x7654u : 0x5432u;
        w.fa = half_bits_to_float(a ? (wd[0] >> 16) : wd[0]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t q = realign(wd[k], wd[k + 1], sel);
            w.c[k] = q & 0x0f0f0f0fu;             // elements 4k..4k+3
            w.c[4 + k] = (q >> 4) & 0x0f0f0f0fu;  // elements 16+4k..
        }
    }
    __device__ __forceinline__ static int idot(const WUnit &w, const XUnit &x) {
        int s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) s = dp4a(w.c[k], x.q[k], s);
        return s - 8 * x.s;
    }
    __device__ __forceinline__ static float accum(float acc, const WUnit &w, int dot, const XUnit &x) {
        return fmaf(w.fa * x.d, (float)dot, acc);
    }
};

// ------------------------------------------------------------------------------- Q4_K / Q5_K
// 6-bit scale S_j and min M_j of sub-block j from the 12 packed bytes (words h1..h3).
__device__ __forceinline__ void kq_scale_min(uint32_t h1, uint32_t h2, uint32_t h3, int j, int &S, int &M) {
    const int sh = 8 * (j & 3);
    const int b0 = (h1 >> sh) & 255, b1 = (h2 >> sh) & 255, b2 = (h3 >> sh) & 255;
    if (j < 4) {
        S = b0 & 63;
        M = b1 & 63;
    } else {
        S = (b2 & 15) | ((b0 >> 6) << 4);
        M = (b2 >> 4) | ((b1 >> 6) << 4);
    }
}

template <int FMT>
struct FmtKQ {
    static constexpr int QK = 256, BS = (FMT == F_Q4_K ? 144 : 176), UPB = 8;
    static constexpr bool NEED_XS = true;
    __device__ __forceinline__ static void decode(uint32_t blk, int j, WUnit &w) {
        const uint4 h = lds128(blk);
        const uint32_t qs = blk + (FMT == F_Q4_K ? 16 : 48) + 32 * (j >> 1);
        const uint4 q0 = lds128(qs), q1 = lds128(qs + 16);
        int S, M;
        kq_scale_min(h.y, h.z, h.w, j, S, M);
        w.fa = half_bits_to_float(h.x) * (float)S;
        w.fb = half_bits_to_float(h.x >> 16) * (float)M;
        const int sh = 4 * (j & 1);
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) w.c[k] = (qw[k] >> sh) & 0x0f0f0f0fu;
        if (FMT == F_Q5_K) {
            const uint4 h0 = lds128(blk + 16), h1 = lds128(blk + 32);
            const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) w.c[k] |= ((hw[k] >> j) & 0x01010101u) << 4;
        }
    }
    __device__ __forceinline__ static int idot(const WUnit &w, const XUnit &x) {
        int s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) s = dp4a(w.c[k], x.q[k], s);
        return s;
    }
    __device__ __forceinline__ static float accum(float acc, const WUnit &w, int dot, const XUnit &x) {
        return fmaf(x.d, fmaf(w.fa, (float)dot, -w.fb * (float)x.s), acc);
    }
};
template <>
struct Fmt<F_Q4_K> : FmtKQ<F_Q4_K> {};
template <>
struct Fmt<F_Q5_K> : FmtKQ<F_Q5_K> {};

// ------------------------------------------------------------------------------- Q6_K
template <>
struct Fmt<F_Q6_K> {
    static constexpr int QK = 256, BS = 210, UPB = 8;
    static constexpr bool NEED_XS = false;
    // unit ut = activation block 4h+t of the superblock: elements 128h + 32t + l, l < 32
    __device__ __forceinline__ static void decode(uint32_t blk, int ut, WUnit &w) {
        const uint32_t a = blk & 3u, base = blk - a;
        const int h = ut >> 2, t = ut & 3;
        const uint32_t sel = a ? 0x7654u : 0x5432u;
        const uint32_t lq = base + 64 * h + 32 * (t & 1);
        const uint32_t hq = base + 128 + 32 * h;
        uint32_t lw[9], hw[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            lw[k] = lds32(lq + 4 * k);
            hw[k] = lds32(hq + 4 * k);
        }
        const int sh = 4 * (t >> 1), hs = 2 * t;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t l = (realign(lw[k], lw[k + 1], sel) >> sh) & 0x0f0f0f0fu;
            const uint32_t hi = (realign(hw[k], hw[k + 1], sel) >> hs) & 0x03030303u;
            // per byte: (l | hi<<4) - 32, done without borrows between bytes
            w.c[k] = ((l | (hi << 4)) + 0x60606060u) ^ 0x80808080u;
        }
        const uint32_t so = a + 192 + 8 * h + 2 * t;  // even
        const uint32_t sw = lds32(base + (so & ~3u)) >> (8 * (so & 3u));
        w.sA = (int)(int8_t)(sw & 255u);
        w.sB = (int)(int8_t)((sw >> 8) & 255u);
        w.fa = half_bits_to_float(lds32(base + 208) >> (8 * a));
    }
    __device__ __forceinline__ static int idot(const WUnit &w, const XUnit &x) {
        int lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) lo = dp4a(w.c[k], x.q[k], lo);
#pragma unroll
        for (int k = 4; k < 8; ++k) hi = dp4a(w.c[k], x.q[k], hi);
        return w.sA * lo + w.sB * hi;
    }
    __device__ __forceinline__ static float accum(float acc, const WUnit &w, int dot, const XUnit &x) {
        return fmaf(w.fa * x.d, (float)dot, acc);
    }
};

// ------------------------------------------------------------------------------- IQ4_XS
constexpr int8_t kIQ4Codebook[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                     1,    13,   25,  38,  53,  69,  89,  113};
constexpr uint32_t cb_word(int i) {
    return (uint32_t)(uint8_t)kIQ4Codebook[i] | ((uint32_t)(uint8_t)kIQ4Codebook[i + 1] << 8) |
           ((uint32_t)(uint8_t)kIQ4Codebook[i + 2] << 16) | ((uint32_t)(uint8_t)kIQ4Codebook[i + 3] << 24);
}

// Codebook lookup of the four 4-bit indices in bits 15:0 of s (one per nibble): two byte
// permutes over the table halves, then a third that keeps, per byte, the half chosen by the
// index's bit 3.
__device__ __forceinline__ uint32_t cb_lookup4(uint32_t s) {
    const uint32_t lo = prmt(cb_word(0), cb_word(4), s & 0x7777u);
    const uint32_t hi = prmt(cb_word(8), cb_word(12), s & 0x7777u);
    return prmt(lo, hi, ((s >> 1) & 0x4444u) | 0x3210u);
}

template <>
struct Fmt<F_IQ4_XS> {
    static constexpr int QK = 256, BS = 136, UPB = 8;
    static constexpr bool NEED_XS = false;
    __device__ __forceinline__ static void decode(uint32_t blk, int ib, WUnit &w) {
        const uint2 hdr = lds64(blk);  // x: d | scales_h << 16, y: scales_l[0..3]
        const uint2 qa = lds64(blk + 8 + 16 * ib), qb = lds64(blk + 16 + 16 * ib);
        const int ls = ((hdr.y >> (4 * ib)) & 15) | (((hdr.x >> (16 + 2 * ib)) & 3) << 4);
        w.fa = half_bits_to_float(hdr.x) * (float)(ls - 32);
        const uint32_t qw[4] = {qa.x, qa.y, qb.x, qb.y};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // nibbles of bytes 0,1 then 2,3: (lo b0, hi b0, lo b1, hi b1)
            const uint32_t A = cb_lookup4(qw[k]);
            const uint32_t B = cb_lookup4(qw[k] >> 16);
            w.c[k] = prmt(A, B, 0x6420u);      // elements 4k..4k+3 (low nibbles)
            w.c[4 + k] = prmt(A, B, 0x7531u);  // elements 16+4k.. (high nibbles)
        }
    }
    __device__ __forceinline__ static int idot(const WUnit &w, const XUnit &x) {
        int s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) s = dp4a(w.c[k], x.q[k], s);
        return s;
    }
    __device__ __forceinline__ static float accum(float acc, const WUnit &w, int dot, const XUnit &x) {
        return fmaf(w.fa * x.d, (float)dot, acc);
    }
};

// ------------------------------------------------------------------------------- activations
// Activation codes in shared memory: q at byte ldq*m + 32*xb, d/s at 4*(lds*m + xb).
struct XSmem {
    uint32_t q, d, s;
    int ldq, lds;
    __device__ __forceinline__ void load(int m, int xb, bool need_s, XUnit &x) const {
        const uint32_t qa = q + (uint32_t)(m * ldq + 32 * xb);
        const uint4 a = lds128(qa), b = lds128(qa + 16);
        x.q[0] = a.x; x.q[1] = a.y; x.q[2] = a.z; x.q[3] = a.w;
        x.q[4] = b.x; x.q[5] = b.y; x.q[6] = b.z; x.q[7] = b.w;
        x.d = __uint_as_float(lds32(d + 4u * (uint32_t)(m * lds + xb)));
        x.s = need_s ? (int)lds32(s + 4u * (uint32_t)(m * lds + xb)) : 0;
    }
};

// Activation codes in global memory (read-only for the kernel's lifetime).
struct XGlob {
    const int8_t *q;
    const float *d;
    const int32_t *s;
    int ldq, lds;
    __device__ __forceinline__ void load(int m, int xb, bool need_s, XUnit &x) const {
        const int8_t *qa = q + (size_t)m * ldq + 32 * (size_t)xb;
        const uint4 a = ldg128_nc(qa), b = ldg128_nc(qa + 16);
        x.q[0] = a.x; x.q[1] = a.y; x.q[2] = a.z; x.q[3] = a.w;
        x.q[4] = b.x; x.q[5] = b.y; x.q[6] = b.z; x.q[7] = b.w;
        x.d = __ldg(d + (size_t)m * lds + xb);
        x.s = need_s ? __ldg(s + (size_t)m * lds + xb) : 0;
    }
};

}  // namespace qg
