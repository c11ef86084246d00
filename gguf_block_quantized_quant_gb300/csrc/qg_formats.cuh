// qg_formats.cuh -- register-resident decoders for the GGUF block formats.
//
// The GEMV is computed on the raw blocks in place ("为什么专家缓存救不了稠密模型", Q&A
// "如何让CUDA直接计算GGUF混合量化块而不展开为FP16？"): weight codes are unpacked in
// registers, multiplied with the int8 activation codes by dp4a into exact int32 sums per
// 32-element unit (one activation block), and the fp32 scale factors are applied to those
// sums (for K-quants together with the min "correction term"; for IQ4_XS after a register
// lookup in the 16-entry codebook).  Byte layouts are the public GGUF block definitions
// (the pages name the formats but do not print them):
//
//   Q8_0    34 B: fp16 d, int8 q[32]                           w = d*q
//   Q4_0    18 B: fp16 d, qs[16]; e<16 low nibble of qs[e],    w = d*(nib-8)
//                 e>=16 high nibble of qs[e-16]
//   Q4_1    20 B: fp16 d, fp16 m, qs[16]                       w = d*nib + m
//   Q5_0    22 B: fp16 d, u32 qh, qs[16] (bit e of qh = 5th)   w = d*(code-16)
//   Q5_1    24 B: fp16 d, fp16 m, u32 qh, qs[16]               w = d*code + m
//   IQ4_NL  18 B: fp16 d, qs[16] codebook indices              w = d*K[idx]
//   Q4_K   144 B: fp16 d, fp16 dmin, sc12[12], qs[128]         w = d*S_j*code - dmin*M_j
//   Q5_K   176 B: fp16 d, fp16 dmin, sc12[12], qh[32], qs[128] (code += 16 * bit j of qh[l])
//   Q6_K   210 B: ql[128], qh[64], int8 sc[16], fp16 d          w = d*sc[e/16]*(code-32)
//   IQ4_XS 136 B: fp16 d, u16 scales_h, scales_l[4], qs[128]   w = d*(ls-32)*K[idx]
//
// Work is organised in TASKS, one per lane: eight, four or one Q4_0 / IQ4_NL blocks, four
// or one Q8_0 / Q4_1 / Q5_0 / Q5_1 blocks, two or one Q4_K / IQ4_XS superblocks, a whole
// Q5_K / Q6_K superblock.  A task's weights are read from shared memory; its activations come from a
// per-task tile (codes, scales d, sums s, packed 16-element half sums and d*s of each
// activation block), padded so that the 16-byte loads of 8 consecutive lanes hit distinct
// banks.  Every unit's dot product is an exact int32 sum; the test-hook sink receives
// those integers (sink.unit), the GEMV sink the benchmark's fp32 contribution to y (sink.add),
// formed with as few conversions and multiplies per unit as the format allows.
#pragma once

#include "qg_common.cuh"

namespace qg {

enum : int {
    F_Q4_0 = 2, F_Q4_1 = 3, F_Q5_0 = 6, F_Q5_1 = 7, F_Q8_0 = 8,
    F_Q2_K = 10, F_Q3_K = 11, F_Q4_K = 12, F_Q5_K = 13, F_Q6_K = 14, F_IQ4_NL = 20, F_IQ4_XS = 23
};

// unsigned (weights) x signed (activations) 4-way byte dot product
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int r;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
__device__ __forceinline__ float ldsf(uint32_t a) { return __uint_as_float(lds32(a)); }

// Shared-memory operands of the decoders are plain pointers derived from the kernel's
// extern __shared__ array: the compiler emits shared loads with immediate offsets and
// schedules them freely between the barrier waits (whose "memory" clobbers order them).
using SAddr = const uint8_t *;
__device__ __forceinline__ uint32_t lds32(SAddr p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint2 lds64(SAddr p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint4 lds128(SAddr p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ float ldsf(SAddr p) { return *reinterpret_cast<const float *>(p); }

// ---------------------------------------------------------------------------------- tiles
// Activation tile of XGT units: codes[32*XGT] | d[XGT] fp32 | s[XGT] int32 |
// h[XGT] (sum of codes 0..15 in the low 16 bits, 16..31 in the high 16 bits) |
// ds[XGT] fp32 (d * s, the activation side of the K-quant min term), padded to an odd
// number of 16-byte chunks.
__host__ __device__ constexpr int tile_raw(int xgt) { return 48 * xgt; }
__host__ __device__ constexpr int tile_stride(int xgt) {
    return ((tile_raw(xgt) + 15) / 16) % 2 == 1 ? (tile_raw(xgt) + 15) / 16 * 16 : (tile_raw(xgt) + 15) / 16 * 16 + 16;
}
template <int XGT>
struct Tile {
    static constexpr int D = 32 * XGT, S = D + 4 * XGT, H = S + 4 * XGT, Q = H + 4 * XGT, STRIDE = tile_stride(XGT);
};

// Four consecutive 32-bit fields of a tile (d, s, h or ds of units u..u+3, u a multiple
// of 4): one 16-byte load, which keeps the lanes of a quarter-warp on distinct banks (the
// tile stride is an odd number of 16-byte chunks) where 32-bit loads of lanes 8 tiles
// apart would share a bank.
__device__ __forceinline__ void ld4(SAddr a, uint32_t *v) {
    const uint4 p = lds128(a);
    v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
}

__device__ __forceinline__ void ldx8(SAddr a, uint32_t (&x)[8]) {
    const uint4 p = lds128(a), q = lds128(a + 16);
    x[0] = p.x; x[1] = p.y; x[2] = p.z; x[3] = p.w;
    x[4] = q.x; x[5] = q.y; x[6] = q.z; x[7] = q.w;
}

// Activations of one task: tile address of token m is base + m * tok_stride.
struct XT {
    SAddr base;
    uint32_t tok_stride;
    __device__ __forceinline__ SAddr tile(int m) const { return base + (uint32_t)m * tok_stride; }
};

// Byte offset OFF (even) into a run of words: realigned when OFF is 2 mod 4.
template <int NW>
__device__ __forceinline__ uint32_t word_at(const uint32_t (&w)[NW], int off) {
    return (off & 3) ? prmt(w[off >> 2], w[(off >> 2) + 1], 0x5432u) : w[off >> 2];
}

// Byte k of w, zero-extended.
__device__ __forceinline__ int byte_of(uint32_t w, int k) { return (int)((w >> (8 * k)) & 255u); }

// Sinks.  A format calls, per token m:
//   DOTS sinks:   unit(m, u, dot, xs) with the exact int32 dot of unit u and the
//                 activation sum xs (the integer contract of the test hook);
//   value sinks:  add(m, v) with the benchmark's fp32 contribution to y.

// ================================================================================ IQ4 codebook
constexpr int8_t kIQ4Codebook[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                     1,    13,   25,  38,  53,  69,  89,  113};
constexpr uint32_t cb_word(int i) {
    return (uint32_t)(uint8_t)kIQ4Codebook[i] | ((uint32_t)(uint8_t)kIQ4Codebook[i + 1] << 8) |
           ((uint32_t)(uint8_t)kIQ4Codebook[i + 2] << 16) | ((uint32_t)(uint8_t)kIQ4Codebook[i + 3] << 24);
}

// Codebook values of the 8 indices in q (byte k: low nibble = element k of the unit's first
// half, high nibble = element k of its second half): byte permutes over the two table
// halves, then a permute that keeps, per byte, the half chosen by the index's bit 3.
__device__ __forceinline__ void cb_lookup8(uint32_t q, uint32_t &lo, uint32_t &hi) {
    const uint32_t i7 = q & 0x77777777u;
    const uint32_t pick = ((q >> 1) & 0x44444444u) | 0x32103210u;
    const uint32_t a0 = prmt(cb_word(0), cb_word(4), i7), b0 = prmt(cb_word(8), cb_word(12), i7);
    const uint32_t a1 = prmt(cb_word(0), cb_word(4), i7 >> 16), b1 = prmt(cb_word(8), cb_word(12), i7 >> 16);
    const uint32_t A = prmt(a0, b0, pick);        // values of nibbles (lo b0, hi b0, lo b1, hi b1)
    const uint32_t B = prmt(a1, b1, pick >> 16);  // values of nibbles (lo b2, hi b2, lo b3, hi b3)
    lo = prmt(A, B, 0x6420u);
    hi = prmt(A, B, 0x7531u);
}

// ====================================================================== 32-element blocks
// Q8_0, Q4_0, Q4_1, Q5_0, Q5_1 and IQ4_NL: T blocks per task.  With T == 4, 8 or 16 every
// block's field offsets are compile-time (a task starts 8-byte, with T >= 8 16-byte,
// aligned); with T == 1 a block may start on any even byte and its fields are realigned
// with run-time byte permutes.  A 16-block (Q4_0) task is held as two halves of 8 blocks.  Every decoder works in two phases: load() copies the
// task's bytes from shared memory into registers (so that the engine can refill the ring
// slot at once), compute() decodes them against the activation tiles.
//
//   Q8_0    34 B: d, q[32]                      dot = sum q*x
//   Q4_0    18 B: d, qs[16]                     dot = sum (nib-8)*x
//   Q4_1    20 B: d, m, qs[16]                  y += d*xd*sum(nib*x) + m*(xd*s)
//   Q5_0    22 B: d, qh[4], qs[16]              dot = sum ((nib|bit<<4)-16)*x
//   Q5_1    24 B: d, m, qh[4], qs[16]           y += d*xd*sum((nib|bit<<4)*x) + m*(xd*s)
//   IQ4_NL  18 B: d, qs[16] (codebook indices)  dot = sum K[idx]*x
// Element e < 16 uses the low nibble of qs[e], e >= 16 the high nibble of qs[e-16]; the
// fifth bit of element e is bit e of the little-endian 32-bit qh.

// Bit i of t (i < 4) moved to bit 4 of byte i.
__device__ __forceinline__ uint32_t spread4_bit4(uint32_t t) { return ((t * 0x00204081u) & 0x01010101u) << 4; }

template <int FMT, int T>
struct FmtLegacy {
    static constexpr int QK = 32, XGT = T, TPB = 1, BPT = T;
    static constexpr int BS = FMT == F_Q8_0 ? 34 : FMT == F_Q4_1 ? 20 : FMT == F_Q5_0 ? 22 : FMT == F_Q5_1 ? 24 : 18;
    static constexpr bool HAS_M = FMT == F_Q4_1 || FMT == F_Q5_1;
    static constexpr bool HAS_QH = FMT == F_Q5_0 || FMT == F_Q5_1;
    static constexpr int QH_OFF = FMT == F_Q5_1 ? 4 : 2;
    static constexpr int QS_OFF = FMT == F_Q4_1 ? 4 : FMT == F_Q5_0 ? 6 : FMT == F_Q5_1 ? 8 : 2;
    static constexpr int NQW = FMT == F_Q8_0 ? 8 : 4;  // code words per block
    static constexpr int TASK_BYTES = T * BS;
    static_assert(T != 16 || FMT == F_Q4_0 || FMT == F_IQ4_NL, "16-block tasks are Q4_0 and IQ4_NL only");
    // T >= 4: per half, its words plus two (the last block's realignment reads past its
    // end); T == 1: the words that cover the block from its 4-byte-aligned start
    // two halves (loaded in swapped order by every other group of 4 lanes): 16-block Q4_0 and
    // 8-block Q4_1 / Q5_1 tasks, whose lane stride is an even number of 16-byte chunks
    static constexpr int NH = (T == 16 || (T == 8 && (FMT == F_Q4_1 || FMT == F_Q5_1))) ? 2 : 1, HB = T / NH;
    static constexpr int HW = HB * BS / 4 + 2;
    static constexpr int WW = T >= 4 ? NH * HW : BS / 4 + 2;

    // With 16 blocks per task the tasks of consecutive lanes are 288 bytes (18 chunks of 16
    // bytes) apart, so lanes l and l + 4 would hit the same banks on every 16-byte load;
    // lanes with bit 2 set load their second half first (a 9-chunk shift), so w[0..HW-1]
    // holds half swap() and w[HW..] the other one.
    __device__ __forceinline__ static int swap() { return NH == 2 ? (int)((threadIdx.x >> 2) & 1) : 0; }

    __device__ __forceinline__ static void load(SAddr addr, uint32_t (&w)[WW]) {
        if constexpr (NH == 2) {
            const int sw = swap();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const SAddr hb = addr + (HB * BS) * (h ^ sw);
#pragma unroll
                for (int i = 0; i < HB * BS / 16; ++i) {
                    const uint4 v = lds128(hb + 16 * i);
                    w[HW * h + 4 * i] = v.x; w[HW * h + 4 * i + 1] = v.y;
                    w[HW * h + 4 * i + 2] = v.z; w[HW * h + 4 * i + 3] = v.w;
                }
                const uint2 v = lds64(hb + HB * BS);
                w[HW * h + HW - 2] = v.x;
                w[HW * h + HW - 1] = v.y;
            }
        } else if constexpr (T == 8) {
#pragma unroll
            for (int i = 0; i < TASK_BYTES / 16; ++i) {
                const uint4 v = lds128(addr + 16 * i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
            const uint2 v = lds64(addr + TASK_BYTES);
            w[WW - 2] = v.x;
            w[WW - 1] = v.y;
        } else if constexpr (T == 4) {
#pragma unroll
            for (int i = 0; i < WW / 2; ++i) {
                const uint2 v = lds64(addr + 8 * i);
                w[2 * i] = v.x;
                w[2 * i + 1] = v.y;
            }
        } else {
            const SAddr base = addr - ((uintptr_t)addr & 3u);
#pragma unroll
            for (int i = 0; i < WW; ++i) w[i] = lds32(base + 4 * i);
        }
    }

    // The 4 bytes at byte offset o (even, compile-time) of a block that starts a (0 or 2)
    // bytes into w[0]: pair (w[o/4], w[o/4+1]) starting at byte a + o%4 of the pair.
    __device__ __forceinline__ static uint32_t rword(const uint32_t (&w)[WW], uint32_t a, int o) {
        return prmt(w[o >> 2], w[(o >> 2) + 1], 0x3210u + 0x2222u * ((a + (uint32_t)(o & 3)) >> 1));
    }

    // Whether a unit needs the activation sum s: the code offset of Q4_0 and Q5_0 is
    // applied through it, and the test hook reports it for the additive-min formats.
    template <class Sink>
    static constexpr bool needs_s() { return FMT == F_Q4_0 || FMT == F_Q5_0 || (Sink::DOTS && HAS_M); }

    // One block against token m's tile, unit u; xd, xs, xq: the unit's activation d, s, ds.
    template <class Sink>
    __device__ __forceinline__ static void unit(const uint32_t (&c)[8], uint32_t qh, float d, float mv, int m, int u,
                                                SAddr tile, float xd, int xs, float xq, Sink &sink) {
        uint32_t x[8];
        ldx8(tile + 32 * u, x);
        const int dot = unit_dot(c, qh, x, xs);
        if constexpr (Sink::DOTS) {
            sink.unit(m, u, dot, xs);
        } else {
            float v = d * xd * (float)dot;
            if constexpr (HAS_M) v = fmaf(mv, xq, v);
            sink.add(m, v);
        }
    }

    // The exact integer dot of one block (codes c, fifth bits qh) with activation codes x
    // (sum xs), the format's code offset included.
    __device__ __forceinline__ static int unit_dot(const uint32_t (&c)[8], uint32_t qh, const uint32_t (&x)[8],
                                                   int xs) {
        int dot = 0;
        if constexpr (FMT == F_Q8_0) {
#pragma unroll
            for (int k = 0; k < 8; ++k) dot = dp4a(c[k], x[k], dot);
        } else if constexpr (FMT == F_Q4_0 || FMT == F_Q4_1) {
            int lo = 0, hi = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                lo = dp4a(c[k] & 0x0f0f0f0fu, x[k], lo);
                hi = dp4a_us(c[k] & 0xf0f0f0f0u, x[4 + k], hi);
            }
            dot = lo + (hi >> 4);
            if constexpr (FMT == F_Q4_0) dot -= 8 * xs;
        } else if constexpr (HAS_QH) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lo = (c[k] & 0x0f0f0f0fu) | spread4_bit4((qh >> (4 * k)) & 15u);
                const uint32_t hi = ((c[k] >> 4) & 0x0f0f0f0fu) | spread4_bit4((qh >> (16 + 4 * k)) & 15u);
                dot = dp4a(lo, x[k], dot);
                dot = dp4a(hi, x[4 + k], dot);
            }
            if constexpr (FMT == F_Q5_0) dot -= 16 * xs;
        } else {  // IQ4_NL
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t lo, hi;
                cb_lookup8(c[k], lo, hi);
                dot = dp4a(lo, x[k], dot);
                dot = dp4a(hi, x[4 + k], dot);
            }
        }
        return dot;
    }

    // Two rows' tasks of the same columns (w0: row 0, w1: row 1; T = 4 or 8 blocks each)
    // against the same activation tiles: every activation load serves both rows.  Per row
    // the arithmetic and its order are compute()'s.
    template <class PSink>
    __device__ __forceinline__ static void compute_pair(const uint32_t (&w0)[WW], uint32_t, const uint32_t (&w1)[WW],
                                                        uint32_t, const XT &xt, int ntok, PSink &sink) {
        static_assert(T == 4 || T == 8, "row pairs take 4- or 8-block tasks");
        using TL = Tile<XGT>;
#pragma unroll
        for (int g = 0; g < T / 4; ++g) {
            float d[2][4], mv[2][4];
            uint32_t qh[2][4], c[2][4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int off = BS * (4 * g + i);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t(&w)[WW] = r ? w1 : w0;
                    d[r][i] = half_bits_to_float((off & 3) ? (w[off >> 2] >> 16) : w[off >> 2]);
                    mv[r][i] = HAS_M ? half_bits_to_float(word_at(w, off + 2)) : 0.0f;
                    qh[r][i] = HAS_QH ? word_at(w, off + QH_OFF) : 0u;
#pragma unroll
                    for (int k = 0; k < NQW; ++k) c[r][i][k] = word_at(w, off + QS_OFF + 4 * k);
                }
            }
            const int u0 = 4 * g;
#pragma unroll
            for (int m = 0; m < PSink::MT; ++m) {
                if (m < ntok) {
                    const SAddr tl = xt.tile(m);
                    uint32_t xd[4], xs[4] = {0u, 0u, 0u, 0u}, xq[4] = {0u, 0u, 0u, 0u};
                    ld4(tl + TL::D + 4 * u0, xd);
                    if constexpr (FMT == F_Q4_0 || FMT == F_Q5_0) ld4(tl + TL::S + 4 * u0, xs);
                    if constexpr (HAS_M) ld4(tl + TL::Q + 4 * u0, xq);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t x[8];
                        ldx8(tl + 32 * (u0 + i), x);
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const int dot = unit_dot(c[r][i], qh[r][i], x, (int)xs[i]);
                            float v = d[r][i] * __uint_as_float(xd[i]) * (float)dot;
                            if constexpr (HAS_M) v = fmaf(mv[r][i], __uint_as_float(xq[i]), v);
                            sink.add(r, m, v);
                        }
                    }
                }
            }
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void compute(const uint32_t (&w)[WW], uint32_t a, int, const XT &xt,
                                                   int ntok, Sink &sink) {
        using TL = Tile<XGT>;
        if constexpr (T >= 4) {
            const int sw = swap();
            // groups of 4 blocks (units u0..u0+3 of one half): their activation d, s and ds
            // come in one 16-byte load each per token
#pragma unroll
            for (int g = 0; g < T / 4; ++g) {
                float d[4], mv[4];
                uint32_t qh[4], c[4][8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int b = 4 * g + i, off = 4 * HW * (b / HB) + BS * (b % HB);
                    d[i] = half_bits_to_float((off & 3) ? (w[off >> 2] >> 16) : w[off >> 2]);
                    mv[i] = HAS_M ? half_bits_to_float(word_at(w, off + 2)) : 0.0f;
                    qh[i] = HAS_QH ? word_at(w, off + QH_OFF) : 0u;
#pragma unroll
                    for (int k = 0; k < NQW; ++k) c[i][k] = word_at(w, off + QS_OFF + 4 * k);
                }
                const int u0 = HB * ((4 * g / HB) ^ sw) + (4 * g) % HB;
#pragma unroll
                for (int m = 0; m < Sink::MT; ++m) {
                    if (m < ntok) {
                        const SAddr tl = xt.tile(m);
                        uint32_t xd[4], xs[4] = {0u, 0u, 0u, 0u}, xq[4] = {0u, 0u, 0u, 0u};
                        ld4(tl + TL::D + 4 * u0, xd);
                        if constexpr (needs_s<Sink>()) ld4(tl + TL::S + 4 * u0, xs);
                        if constexpr (HAS_M && !Sink::DOTS) ld4(tl + TL::Q + 4 * u0, xq);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            unit(c[i], qh[i], d[i], mv[i], m, u0 + i, tl, __uint_as_float(xd[i]), (int)xs[i],
                                 __uint_as_float(xq[i]), sink);
                    }
                }
            }
        } else {
            const float d = half_bits_to_float(rword(w, a, 0));
            const float mv = HAS_M ? half_bits_to_float(rword(w, a, 2)) : 0.0f;
            const uint32_t qh = HAS_QH ? rword(w, a, QH_OFF) : 0u;
            uint32_t c[8];
#pragma unroll
            for (int k = 0; k < NQW; ++k) c[k] = rword(w, a, QS_OFF + 4 * k);
#pragma unroll
            for (int m = 0; m < Sink::MT; ++m) {
                if (m < ntok) {
                    const SAddr tl = xt.tile(m);
                    const int xs = needs_s<Sink>() ? (int)lds32(tl + TL::S) : 0;
                    const float xq = HAS_M && !Sink::DOTS ? ldsf(tl + TL::Q) : 0.0f;
                    unit(c, qh, d, mv, m, 0, tl, ldsf(tl + TL::D), xs, xq, sink);
                }
            }
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void run(SAddr addr, int hf, const XT &xt, int ntok, Sink &sink) {
        uint32_t w[WW];
        load(addr, w);
        compute(w, (uint32_t)((uintptr_t)addr & 3u), hf, xt, ntok, sink);
    }
};

// ================================================================================ Q2_K
// T superblocks per task (84 bytes each: 4-byte aligned; a two-superblock task starts
// 8-byte aligned).  Words: 0..3 the 16 scale|min bytes (low nibble: scale, high nibble:
// min of a 16-element sub-block), 4..19 the 2-bit codes, 20 d | dmin << 16.  Activation
// unit u = 4h + j takes bits 2j, 2j+1 of code words 4 + 8h .. 4 + 8h + 7; its first 16
// elements are sub-block 2u, the last 16 sub-block 2u + 1.  Per unit the exact integers
// are D = S_2u * dot(first 16) + S_2u+1 * dot(last 16) and the min sum
// Mn = M_2u * h_lo + M_2u+1 * h_hi (h: the activation half sums of the tile); per token
// A = sum xd * D and B = sum xd * Mn, and y += d * A - dmin * B once per superblock.
template <int T>
struct FmtQ2K {
    static constexpr int QK = 256, BS = 84, XGT = 8 * T, TPB = 1, BPT = T, TASK_BYTES = 84 * T;
    static constexpr int WW = 21 * T;

    __device__ __forceinline__ static void load(SAddr addr, uint32_t (&w)[WW]) {
        if constexpr (T == 2) {
#pragma unroll
            for (int i = 0; i < WW / 2; ++i) {
                const uint2 v = lds64(addr + 8 * i);
                w[2 * i] = v.x;
                w[2 * i + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < WW; ++i) w[i] = lds32(addr + 4 * i);
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void superblock(const uint32_t *w, int u0, const XT &xt, int ntok,
                                                      Sink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = Sink::MT;
        const float d = half_bits_to_float(w[20]), dmin = half_bits_to_float(w[20] >> 16);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= ntok) continue;
            const SAddr t = xt.tile(m);
            uint32_t xd[8], xh[8];
            ld4(t + TL::H + 4 * u0, xh);
            ld4(t + TL::H + 4 * u0 + 16, xh + 4);
            if constexpr (!Sink::DOTS) {
                ld4(t + TL::D + 4 * u0, xd);
                ld4(t + TL::D + 4 * u0 + 16, xd + 4);
            }
            float A = 0.0f, B = 0.0f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int h = u >> 2, j = u & 3;
                const uint32_t sm = (w[u >> 1] >> (16 * (u & 1))) & 0xffffu;  // bytes 2u, 2u+1
                const int sa = (int)(sm & 15u), ma = (int)((sm >> 4) & 15u);
                const int sb = (int)((sm >> 8) & 15u), mb = (int)(sm >> 12);
                uint32_t x[8];
                ldx8(t + 32 * (u0 + u), x);
                // codes masked in place (bytes 4^j * code, unsigned) and the sums shifted
                // back once: exact, every term is a multiple of 4^j
                const uint32_t msk = 0x03030303u << (2 * j);
                int lo = 0, hi = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    lo = dp4a_us(w[4 + 8 * h + k] & msk, x[k], lo);
                    hi = dp4a_us(w[8 + 8 * h + k] & msk, x[4 + k], hi);
                }
                lo >>= 2 * j;
                hi >>= 2 * j;
                const int hlo = (int)(int16_t)(xh[u] & 0xffffu), hhi = (int)(int16_t)(xh[u] >> 16);
                const int D = sa * lo + sb * hi, Mn = ma * hlo + mb * hhi;
                if constexpr (Sink::DOTS) {
                    sink.unit(m, u0 + u, D, Mn);
                } else {
                    A = fmaf(__uint_as_float(xd[u]), (float)D, A);
                    B = fmaf(__uint_as_float(xd[u]), (float)Mn, B);
                }
            }
            if constexpr (!Sink::DOTS) sink.add(m, fmaf(d, A, -dmin * B));
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void compute(const uint32_t (&w)[WW], uint32_t, int, const XT &xt, int ntok,
                                                   Sink &sink) {
#pragma unroll
        for (int i = 0; i < T; ++i) superblock(w + 21 * i, 8 * i, xt, ntok, sink);
    }

    template <class Sink>
    __device__ __forceinline__ static void run(SAddr addr, int hf, const XT &xt, int ntok, Sink &sink) {
        uint32_t w[WW];
        load(addr, w);
        compute(w, 0, hf, xt, ntok, sink);
    }
};

// ================================================================================ Q3_K
// One whole superblock per task (110 bytes, starting on any even byte: the 28 words from
// the 4-byte-aligned start are loaded and realigned with byte permutes).  Block words:
// 0..7 the third code bits (bit 4h + j of byte l for element 128h + 32j + l), 8..23 the
// low 2-bit codes (as Q2_K), 24..26 the sixteen packed 6-bit scales, 27 d.  Codes are used
// unsigned (0..7) and the -4 offset is applied through the activation half sums, so that
// per unit D = sc_2u * (dot_lo - 4 h_lo) + sc_2u+1 * (dot_hi - 4 h_hi) is exact; per token
// A = sum xd * D, y += d * A.
template <int T>
struct FmtQ3K {
    static_assert(T == 2, "Q3_K tasks are whole superblocks");
    static constexpr int QK = 256, BS = 110, XGT = 8, TPB = 1, BPT = 1, TASK_BYTES = 110;
    static constexpr int WW = 28;

    __device__ __forceinline__ static void load(SAddr addr, uint32_t (&w)[WW]) {
        const SAddr base = addr - ((uintptr_t)addr & 3u);
#pragma unroll
        for (int i = 0; i < WW; ++i) w[i] = lds32(base + 4 * i);
    }

    template <class Sink>
    __device__ __forceinline__ static void compute(const uint32_t (&w)[WW], uint32_t a, int, const XT &xt, int ntok,
                                                   Sink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = Sink::MT;
        const uint32_t sel = a ? 0x5432u : 0x3210u;
        auto word = [&](int i) { return prmt(w[i], w[i + 1], sel); };  // block word i (i < 27)
        // the sixteen scales as bytes 0..63 (scale + 32): low nibbles from block bytes 96..103,
        // high 2 bits from bytes 104..107
        const uint32_t s0 = word(24), s1 = word(25), s2 = word(26);
        uint32_t sc[4];
        sc[0] = (s0 & 0x0f0f0f0fu) | ((s2 & 0x03030303u) << 4);
        sc[1] = (s1 & 0x0f0f0f0fu) | (((s2 >> 2) & 0x03030303u) << 4);
        sc[2] = ((s0 >> 4) & 0x0f0f0f0fu) | (((s2 >> 4) & 0x03030303u) << 4);
        sc[3] = ((s1 >> 4) & 0x0f0f0f0fu) | (((s2 >> 6) & 0x03030303u) << 4);
        const float d = half_bits_to_float(a ? (w[27] >> 16) : w[27]);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= ntok) continue;
            const SAddr t = xt.tile(m);
            uint32_t xd[8], xh[8];
            ld4(t + TL::H, xh);
            ld4(t + TL::H + 16, xh + 4);
            if constexpr (!Sink::DOTS) {
                ld4(t + TL::D, xd);
                ld4(t + TL::D + 16, xd + 4);
            }
            float A = 0.0f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int h = u >> 2, j = u & 3;
                uint32_t x[8];
                ldx8(t + 32 * u, x);
                // low 2 bits and third bit each masked in place (bytes 4^j * bits and
                // 2^u * bit, unsigned), their sums shifted back once: exact
                const uint32_t ml = 0x03030303u << (2 * j), mh = 0x01010101u << u;
                int lo = 0, hi = 0, lb = 0, hb = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    lo = dp4a_us(word(8 + 8 * h + k) & ml, x[k], lo);
                    hi = dp4a_us(word(12 + 8 * h + k) & ml, x[4 + k], hi);
                    lb = dp4a_us(word(k) & mh, x[k], lb);
                    hb = dp4a_us(word(4 + k) & mh, x[4 + k], hb);
                }
                lo = (lo >> (2 * j)) + 4 * (lb >> u);
                hi = (hi >> (2 * j)) + 4 * (hb >> u);
                const int hlo = (int)(int16_t)(xh[u] & 0xffffu), hhi = (int)(int16_t)(xh[u] >> 16);
                const int sa = (int)((sc[u >> 1] >> (16 * (u & 1))) & 255u) - 32;
                const int sb = (int)((sc[u >> 1] >> (16 * (u & 1) + 8)) & 255u) - 32;
                const int D = sa * (lo - 4 * hlo) + sb * (hi - 4 * hhi);
                if constexpr (Sink::DOTS) {
                    sink.unit(m, u, D, 0);
                } else {
                    A = fmaf(__uint_as_float(xd[u]), (float)D, A);
                }
            }
            if constexpr (!Sink::DOTS) sink.add(m, d * A);
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void run(SAddr addr, int hf, const XT &xt, int ntok, Sink &sink) {
        uint32_t w[WW];
        load(addr, w);
        compute(w, (uint32_t)((uintptr_t)addr & 3u), hf, xt, ntok, sink);
    }
};

// ================================================================================ Q4_K
// T superblocks per task (16-byte aligned).  The 8 six-bit scales and mins are unpacked four
// at a time into bytes; sub-block 2p uses the low nibbles of qs[32p..32p+31], sub-block 2p+1
// the high nibbles, which are multiplied in place (16 * nibble) by an unsigned dp4a.  Value
// path: per token, A = sum_j xd_j * (S_j * dot_j) and B = sum_j (xd_j * s_j) * M_j are
// accumulated, and the superblock's d and dmin are applied once: y += d * A - dmin * B.
template <int T>
struct FmtQ4K {
    static constexpr int QK = 256, BS = 144, XGT = 8 * T, TPB = 1, BPT = T, TASK_BYTES = 144 * T;
    static constexpr int WW = 36 * T;

    // With two superblocks per task the tasks of consecutive lanes are 288 bytes (18 chunks
    // of 16 bytes) apart, so lanes l and l + 4 would hit the same banks on every 16-byte
    // load; lanes with bit 2 set load their second superblock first (a 9-chunk shift), so
    // w[0..35] holds superblock swap() and w[36..71] the other one.
    __device__ __forceinline__ static int swap() { return T == 2 ? (int)((threadIdx.x >> 2) & 1) : 0; }

    __device__ __forceinline__ static void load(SAddr addr, uint32_t (&w)[WW]) {
        const int sw = swap();
#pragma unroll
        for (int i = 0; i < T; ++i) {
            const SAddr sb = addr + BS * (i ^ sw);
#pragma unroll
            for (int c = 0; c < 9; ++c) {
                const uint4 v = lds128(sb + 16 * c);
                w[36 * i + 4 * c] = v.x; w[36 * i + 4 * c + 1] = v.y;
                w[36 * i + 4 * c + 2] = v.z; w[36 * i + 4 * c + 3] = v.w;
            }
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void superblock(const uint32_t *w, int u0, const XT &xt, int ntok,
                                                      Sink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = Sink::MT;
        const uint32_t S03 = w[1] & 0x3f3f3f3fu, M03 = w[2] & 0x3f3f3f3fu;
        const uint32_t S47 = (w[3] & 0x0f0f0f0fu) | ((w[1] >> 2) & 0x30303030u);
        const uint32_t M47 = ((w[3] >> 4) & 0x0f0f0f0fu) | ((w[2] >> 2) & 0x30303030u);
        const float d = half_bits_to_float(w[0]), dmin = half_bits_to_float(w[0] >> 16);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= ntok) continue;
            const SAddr t = xt.tile(m);
            // the 8 units' activation d and ds: 16-byte loads
            uint32_t xd[8], xq[8];
            if constexpr (!Sink::DOTS) {
                ld4(t + TL::D + 4 * u0, xd);
                ld4(t + TL::D + 4 * u0 + 16, xd + 4);
                ld4(t + TL::Q + 4 * u0, xq);
                ld4(t + TL::Q + 4 * u0 + 16, xq + 4);
            }
            float A = 0.0f, B = 0.0f;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint32_t *q = w + 4 + 8 * p;
                const uint32_t Sw = p < 2 ? S03 : S47, Mw = p < 2 ? M03 : M47;
                const int k0 = 2 * (p & 1);
                const int sc0 = byte_of(Sw, k0), sc1 = byte_of(Sw, k0 + 1);
                const float mn0 = (float)byte_of(Mw, k0), mn1 = (float)byte_of(Mw, k0 + 1);
                const int u = u0 + 2 * p;
                {
                    uint32_t xa[8], xb[8];
                    ldx8(t + 32 * u, xa);
                    ldx8(t + 32 * u + 32, xb);
                    int da = 0, db = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        da = dp4a(q[k] & 0x0f0f0f0fu, xa[k], da);
                        db = dp4a_us(q[k] & 0xf0f0f0f0u, xb[k], db);
                    }
                    db >>= 4;
                    if constexpr (Sink::DOTS) {
                        const uint2 xs = lds64(t + TL::S + 4 * u);
                        sink.unit(m, u, da, (int)xs.x);
                        sink.unit(m, u + 1, db, (int)xs.y);
                    } else {
                        A = fmaf(__uint_as_float(xd[2 * p]), (float)(sc0 * da), A);
                        A = fmaf(__uint_as_float(xd[2 * p + 1]), (float)(sc1 * db), A);
                        B = fmaf(__uint_as_float(xq[2 * p]), mn0, B);
                        B = fmaf(__uint_as_float(xq[2 * p + 1]), mn1, B);
                    }
                }
            }
            if constexpr (!Sink::DOTS) sink.add(m, fmaf(d, A, -dmin * B));
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void compute(const uint32_t (&w)[WW], uint32_t, int, const XT &xt, int ntok,
                                                   Sink &sink) {
        const int sw = swap();
#pragma unroll
        for (int i = 0; i < T; ++i) superblock(w + 36 * i, 8 * (i ^ sw), xt, ntok, sink);
    }

    // Two rows' superblocks of the same column (T == 1) against the same activation tile:
    // every activation load serves both rows.  Per row the arithmetic and its order are
    // superblock()'s.
    template <class PSink>
    __device__ __forceinline__ static void compute_pair(const uint32_t (&w0)[WW], uint32_t, const uint32_t (&w1)[WW],
                                                        uint32_t, const XT &xt, int ntok, PSink &sink) {
        static_assert(T == 1, "row pairs take one-superblock tasks");
        using TL = Tile<XGT>;
        constexpr int MT = PSink::MT;
        if constexpr (MT >= 16) {
            compute_pair_tokens_inner(w0, 0u, w1, 0u, xt, ntok, sink);
            return;
        }
        uint32_t S03[2], M03[2], S47[2], M47[2];
        float d[2], dmin[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint32_t(&w)[WW] = r ? w1 : w0;
            S03[r] = w[1] & 0x3f3f3f3fu;
            M03[r] = w[2] & 0x3f3f3f3fu;
            S47[r] = (w[3] & 0x0f0f0f0fu) | ((w[1] >> 2) & 0x30303030u);
            M47[r] = ((w[3] >> 4) & 0x0f0f0f0fu) | ((w[2] >> 2) & 0x30303030u);
            d[r] = half_bits_to_float(w[0]);
            dmin[r] = half_bits_to_float(w[0] >> 16);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= ntok) continue;
            const SAddr t = xt.tile(m);
            uint32_t xd[8], xq[8];
            ld4(t + TL::D, xd);
            ld4(t + TL::D + 16, xd + 4);
            ld4(t + TL::Q, xq);
            ld4(t + TL::Q + 16, xq + 4);
            float A[2] = {0.0f, 0.0f}, B[2] = {0.0f, 0.0f};
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t xa[8], xb[8];
                ldx8(t + 64 * p, xa);
                ldx8(t + 64 * p + 32, xb);
                const int k0 = 2 * (p & 1);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t(&w)[WW] = r ? w1 : w0;
                    const uint32_t *q = w + 4 + 8 * p;
                    const uint32_t Sw = p < 2 ? S03[r] : S47[r], Mw = p < 2 ? M03[r] : M47[r];
                    int da = 0, db = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        da = dp4a(q[k] & 0x0f0f0f0fu, xa[k], da);
                        db = dp4a_us(q[k] & 0xf0f0f0f0u, xb[k], db);
                    }
                    db >>= 4;
                    A[r] = fmaf(__uint_as_float(xd[2 * p]), (float)(byte_of(Sw, k0) * da), A[r]);
                    A[r] = fmaf(__uint_as_float(xd[2 * p + 1]), (float)(byte_of(Sw, k0 + 1) * db), A[r]);
                    B[r] = fmaf(__uint_as_float(xq[2 * p]), (float)byte_of(Mw, k0), B[r]);
                    B[r] = fmaf(__uint_as_float(xq[2 * p + 1]), (float)byte_of(Mw, k0 + 1), B[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) sink.add(r, m, fmaf(d[r], A[r], -dmin[r] * B[r]));
        }
    }

    // compute_pair with the loop over unit pairs outside and tokens inside (16 tokens per
    // lane): a unit's masked code words and its scales folded with d and dmin (fp32) are
    // formed once for all tokens, and per token and row a unit pair costs its 16 dp4a, two
    // conversions and four FMAs into the row's sum.  Measured 17 % faster than the
    // token-outer order at 16 tokens, equal at 8 and slower at 2 and 4.
    template <class PSink>
    __device__ __forceinline__ static void compute_pair_tokens_inner(const uint32_t (&w0)[WW], uint32_t, const uint32_t (&w1)[WW],
                                                        uint32_t, const XT &xt, int ntok, PSink &sink) {
        static_assert(T == 1, "row pairs take one-superblock tasks");
        using TL = Tile<XGT>;
        constexpr int MT = PSink::MT;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int k0 = 2 * (p & 1);
            uint32_t lo[2][8], hi[2][8];
            float dsc[2][2], dmn[2][2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t(&w)[WW] = r ? w1 : w0;
                const uint32_t Sw = p < 2 ? (w[1] & 0x3f3f3f3fu) : ((w[3] & 0x0f0f0f0fu) | ((w[1] >> 2) & 0x30303030u));
                const uint32_t Mw =
                    p < 2 ? (w[2] & 0x3f3f3f3fu) : (((w[3] >> 4) & 0x0f0f0f0fu) | ((w[2] >> 2) & 0x30303030u));
                const float d = half_bits_to_float(w[0]), dmin = half_bits_to_float(w[0] >> 16);
                dsc[r][0] = d * (float)byte_of(Sw, k0);
                dsc[r][1] = d * (float)byte_of(Sw, k0 + 1);
                dmn[r][0] = dmin * (float)byte_of(Mw, k0);
                dmn[r][1] = dmin * (float)byte_of(Mw, k0 + 1);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    lo[r][k] = w[4 + 8 * p + k] & 0x0f0f0f0fu;
                    hi[r][k] = w[4 + 8 * p + k] & 0xf0f0f0f0u;
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m >= ntok) continue;
                const SAddr t = xt.tile(m);
                uint32_t xa[8], xb[8];
                ldx8(t + 64 * p, xa);
                ldx8(t + 64 * p + 32, xb);
                const uint2 xd = lds64(t + TL::D + 8 * p), xq = lds64(t + TL::Q + 8 * p);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    int da = 0, db = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        da = dp4a(lo[r][k], xa[k], da);
                        db = dp4a_us(hi[r][k], xb[k], db);
                    }
                    db >>= 4;
                    float v = sink.acc[r][m];
                    v = fmaf((float)da, __uint_as_float(xd.x) * dsc[r][0], v);
                    v = fmaf((float)db, __uint_as_float(xd.y) * dsc[r][1], v);
                    v = fmaf(-__uint_as_float(xq.x), dmn[r][0], v);
                    v = fmaf(-__uint_as_float(xq.y), dmn[r][1], v);
                    sink.acc[r][m] = v;
                }
            }
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void run(SAddr addr, int hf, const XT &xt, int ntok, Sink &sink) {
        uint32_t w[WW];
        load(addr, w);
        compute(w, 0, hf, xt, ntok, sink);
    }
};

// ================================================================================ Q5_K
// One whole superblock per task (16-byte aligned).  The fifth bit of sub-block j is bit j
// of each qh byte.  Combine as Q4_K.
template <int T>
struct FmtQ5K {
    static_assert(T == 2, "Q5_K tasks are whole superblocks");
    static constexpr int QK = 256, BS = 176, XGT = 8, TPB = 1, BPT = 1, TASK_BYTES = 176;
    static constexpr int WW = 44;

    __device__ __forceinline__ static void load(SAddr addr, uint32_t (&w)[WW]) {
#pragma unroll
        for (int c = 0; c < 11; ++c) {
            const uint4 v = lds128(addr + 16 * c);
            w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void compute(const uint32_t (&w)[WW], uint32_t, int, const XT &xt, int ntok,
                                                   Sink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = Sink::MT;
        const uint32_t *qh = w + 4;
        const float d = half_bits_to_float(w[0]), dmin = half_bits_to_float(w[0] >> 16);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= ntok) continue;
            const SAddr t = xt.tile(m);
            // the 8 units' activation d and ds: 16-byte loads
            uint32_t xd[8], xq[8];
            if constexpr (!Sink::DOTS) {
                ld4(t + TL::D, xd);
                ld4(t + TL::D + 16, xd + 4);
                ld4(t + TL::Q, xq);
                ld4(t + TL::Q + 16, xq + 4);
            }
            float A = 0.0f, B = 0.0f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t Sw = hf ? ((w[3] & 0x0f0f0f0fu) | ((w[1] >> 2) & 0x30303030u)) : (w[1] & 0x3f3f3f3fu);
                const uint32_t Mw =
                    hf ? (((w[3] >> 4) & 0x0f0f0f0fu) | ((w[2] >> 2) & 0x30303030u)) : (w[2] & 0x3f3f3f3fu);
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const int j0 = 4 * hf + 2 * pp;  // sub-blocks j0 (low nibbles) and j0+1 (high nibbles)
                    const uint32_t *q = w + 12 + 8 * (2 * hf + pp);
                    const int sc0 = byte_of(Sw, 2 * pp), sc1 = byte_of(Sw, 2 * pp + 1);
                    const float mn0 = (float)byte_of(Mw, 2 * pp), mn1 = (float)byte_of(Mw, 2 * pp + 1);
                    uint32_t xa[8], xb[8];
                    ldx8(t + 32 * j0, xa);
                    ldx8(t + 32 * j0 + 32, xb);
                    // nibbles and fifth bits masked where they sit (unsigned bytes), each sum
                    // shifted back once: exact, every term is a multiple of the bit weight
                    const uint32_t ma = 0x01010101u << j0, mb = 0x01010101u << (j0 + 1);
                    int la = 0, lb = 0, ha = 0, hb = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        la = dp4a_us(q[k] & 0x0f0f0f0fu, xa[k], la);
                        lb = dp4a_us(q[k] & 0xf0f0f0f0u, xb[k], lb);
                        ha = dp4a_us(qh[k] & ma, xa[k], ha);
                        hb = dp4a_us(qh[k] & mb, xb[k], hb);
                    }
                    const int da = la + 16 * (ha >> j0), db = (lb >> 4) + 16 * (hb >> (j0 + 1));
                    if constexpr (Sink::DOTS) {
                        const uint2 xs = lds64(t + TL::S + 4 * j0);
                        sink.unit(m, j0, da, (int)xs.x);
                        sink.unit(m, j0 + 1, db, (int)xs.y);
                    } else {
                        A = fmaf(__uint_as_float(xd[j0]), (float)(sc0 * da), A);
                        A = fmaf(__uint_as_float(xd[j0 + 1]), (float)(sc1 * db), A);
                        B = fmaf(__uint_as_float(xq[j0]), mn0, B);
                        B = fmaf(__uint_as_float(xq[j0 + 1]), mn1, B);
                    }
                }
            }
            if constexpr (!Sink::DOTS) sink.add(m, fmaf(d, A, -dmin * B));
        }
    }

    // Two rows' superblocks of the same column against the same activation tile (every
    // activation load serves both rows); per row the arithmetic and its order are compute()'s.
    template <class PSink>
    __device__ __forceinline__ static void compute_pair(const uint32_t (&w0)[WW], uint32_t, const uint32_t (&w1)[WW],
                                                        uint32_t, const XT &xt, int ntok, PSink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = PSink::MT;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= ntok) continue;
            const SAddr t = xt.tile(m);
            uint32_t xd[8], xq[8];
            ld4(t + TL::D, xd);
            ld4(t + TL::D + 16, xd + 4);
            ld4(t + TL::Q, xq);
            ld4(t + TL::Q + 16, xq + 4);
            float A[2] = {0.0f, 0.0f}, B[2] = {0.0f, 0.0f};
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const int j0 = 4 * hf + 2 * pp;
                    uint32_t xa[8], xb[8];
                    ldx8(t + 32 * j0, xa);
                    ldx8(t + 32 * j0 + 32, xb);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const uint32_t(&w)[WW] = r ? w1 : w0;
                        const uint32_t *qh = w + 4;
                        const uint32_t Sw =
                            hf ? ((w[3] & 0x0f0f0f0fu) | ((w[1] >> 2) & 0x30303030u)) : (w[1] & 0x3f3f3f3fu);
                        const uint32_t Mw =
                            hf ? (((w[3] >> 4) & 0x0f0f0f0fu) | ((w[2] >> 2) & 0x30303030u)) : (w[2] & 0x3f3f3f3fu);
                        const uint32_t *q = w + 12 + 8 * (2 * hf + pp);
                        int da = 0, db = 0;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            da = dp4a((q[k] & 0x0f0f0f0fu) | (((qh[k] >> j0) & 0x01010101u) << 4), xa[k], da);
                            db = dp4a(((q[k] >> 4) & 0x0f0f0f0fu) | (((qh[k] >> (j0 + 1)) & 0x01010101u) << 4), xb[k],
                                      db);
                        }
                        A[r] = fmaf(__uint_as_float(xd[j0]), (float)(byte_of(Sw, 2 * pp) * da), A[r]);
                        A[r] = fmaf(__uint_as_float(xd[j0 + 1]), (float)(byte_of(Sw, 2 * pp + 1) * db), A[r]);
                        B[r] = fmaf(__uint_as_float(xq[j0]), (float)byte_of(Mw, 2 * pp), B[r]);
                        B[r] = fmaf(__uint_as_float(xq[j0 + 1]), (float)byte_of(Mw, 2 * pp + 1), B[r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t(&w)[WW] = r ? w1 : w0;
                sink.add(r, m, fmaf(half_bits_to_float(w[0]), A[r], -half_bits_to_float(w[0] >> 16) * B[r]));
            }
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void run(SAddr addr, int hf, const XT &xt, int ntok, Sink &sink) {
        uint32_t w[WW];
        load(addr, w);
        compute(w, 0, hf, xt, ntok, sink);
    }
};

// ================================================================================ Q6_K
// One whole superblock per task.  Within half hf, activation block t = 0..3: the low four
// bits of element 32t + l come from byte l + 32*(t&1) of the half's 64 ql bytes (low nibble
// for t < 2), the top two from bits 2t, 2t+1 of qh byte l.  Codes are used unsigned (0..63)
// and the -32 offset is applied through the activation half sums.  Superblocks start on any
// even byte: the words from the 4-byte-aligned start are loaded and realigned with byte
// permutes.  Value path: sum_t xd_t * dot_t per token, times d once.
template <int T>
struct FmtQ6K {
    static_assert(T == 2, "Q6_K tasks are whole superblocks");
    static constexpr int QK = 256, BS = 210, XGT = 8, TPB = 1, BPT = 1, TASK_BYTES = 210;
    static constexpr int WW = 54;  // 216 bytes from the aligned start cover the block

    __device__ __forceinline__ static void load(SAddr addr, uint32_t (&w)[WW]) {
        const SAddr base = addr - ((uintptr_t)addr & 3u);
#pragma unroll
        for (int i = 0; i < WW; ++i) w[i] = lds32(base + 4 * i);
    }

    template <class Sink>
    __device__ __forceinline__ static void compute(const uint32_t (&w)[WW], uint32_t a, int, const XT &xt, int ntok,
                                                   Sink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = Sink::MT;
        const uint32_t sel = a ? 0x5432u : 0x3210u;
        float A[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) A[m] = 0.0f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t hw[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) hw[k] = prmt(w[32 + 8 * hf + k], w[33 + 8 * hf + k], sel);
            // sub-scales 8hf..8hf+7 start at byte 192 + 8hf of the block
            const uint32_t scA = prmt(w[48 + 2 * hf], w[49 + 2 * hf], sel);  // sc[8hf+0..3]
            const uint32_t scB = prmt(w[49 + 2 * hf], w[50 + 2 * hf], sel);  // sc[8hf+4..7]
            // up to 4 tokens: the half's activation d and h of every token in two 16-byte
            // loads (more tokens: one 32-bit load per unit, to spare registers)
            constexpr bool VEC = MT <= 4;
            uint32_t xdv[VEC ? MT : 1][4], xhv[VEC ? MT : 1][4];
            if constexpr (VEC && !Sink::DOTS) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < ntok) {
                        ld4(xt.tile(m) + TL::D + 16 * hf, xdv[m]);
                        ld4(xt.tile(m) + TL::H + 16 * hf, xhv[m]);
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                uint32_t lw[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) lw[k] = prmt(w[16 * hf + 8 * s + k], w[16 * hf + 8 * s + k + 1], sel);
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int t = s + 2 * tt;  // activation block within the half
                    const int u = 4 * hf + t;  // its unit in the task tile
                    // up to 2 tokens: the low 4 and high 2 code bits masked where they sit
                    // (unsigned bytes) and each sum shifted back once (exact), two dots per
                    // word; more tokens: the 6-bit codes assembled once and one dot per word
                    constexpr bool SPLIT = MT <= 2;
                    uint32_t c[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        c[k] = SPLIT ? 0u
                                     : ((lw[k] >> (4 * tt)) & 0x0f0f0f0fu) | (((hw[k] >> (2 * t)) & 0x03030303u) << 4);
                    const uint32_t scw = t < 2 ? scA : scB;
                    const int sA = (int)(int8_t)((scw >> (16 * (t & 1))) & 255u);
                    const int sB = (int)(int8_t)((scw >> (16 * (t & 1) + 8)) & 255u);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < ntok) {
                            const SAddr tl = xt.tile(m);
                            uint32_t x[8];
                            ldx8(tl + 32 * u, x);
                            const uint32_t xh = VEC && !Sink::DOTS ? xhv[VEC ? m : 0][t] : lds32(tl + TL::H + 4 * u);
                            int lo = 0, hi = 0;
                            if constexpr (SPLIT) {
                                const uint32_t ml = 0x0f0f0f0fu << (4 * tt), mh = 0x03030303u << (2 * t);
                                int l0 = 0, l1 = 0, h0 = 0, h1 = 0;
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    l0 = dp4a_us(lw[k] & ml, x[k], l0);
                                    h0 = dp4a_us(hw[k] & mh, x[k], h0);
                                    l1 = dp4a_us(lw[4 + k] & ml, x[4 + k], l1);
                                    h1 = dp4a_us(hw[4 + k] & mh, x[4 + k], h1);
                                }
                                lo = (l0 >> (4 * tt)) + 16 * (h0 >> (2 * t));
                                hi = (l1 >> (4 * tt)) + 16 * (h1 >> (2 * t));
                            } else {
#pragma unroll
                                for (int k = 0; k < 4; ++k) lo = dp4a(c[k], x[k], lo);
#pragma unroll
                                for (int k = 4; k < 8; ++k) hi = dp4a(c[k], x[k], hi);
                            }
                            const int hlo = (int)(int16_t)(xh & 0xffffu), hhi = (int)(int16_t)(xh >> 16);
                            const int dot = sA * (lo - 32 * hlo) + sB * (hi - 32 * hhi);
                            if constexpr (Sink::DOTS) {
                                sink.unit(m, u, dot, 0);
                            } else {
                                const float xd = VEC ? __uint_as_float(xdv[VEC ? m : 0][t]) : ldsf(tl + TL::D + 4 * u);
                                A[m] = fmaf(xd, (float)dot, A[m]);
                            }
                        }
                    }
                }
            }
        }
        if constexpr (!Sink::DOTS) {
            const float d = half_bits_to_float(w[52] >> (8 * a));
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < ntok) sink.add(m, d * A[m]);
        }
    }

    // Two rows' superblocks of the same column (each with its own 2-byte alignment a0, a1)
    // against the same activation tile; per row the arithmetic and its order are compute()'s.
    template <class PSink>
    __device__ __forceinline__ static void compute_pair(const uint32_t (&w0)[WW], uint32_t a0,
                                                        const uint32_t (&w1)[WW], uint32_t a1, const XT &xt, int ntok,
                                                        PSink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = PSink::MT;
        const uint32_t sel[2] = {a0 ? 0x5432u : 0x3210u, a1 ? 0x5432u : 0x3210u};
        float A[2][MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) A[0][m] = A[1][m] = 0.0f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t hw[2][8], scA[2], scB[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t(&w)[WW] = r ? w1 : w0;
#pragma unroll
                for (int k = 0; k < 8; ++k) hw[r][k] = prmt(w[32 + 8 * hf + k], w[33 + 8 * hf + k], sel[r]);
                scA[r] = prmt(w[48 + 2 * hf], w[49 + 2 * hf], sel[r]);
                scB[r] = prmt(w[49 + 2 * hf], w[50 + 2 * hf], sel[r]);
            }
            constexpr bool VEC = MT <= 4;
            uint32_t xdv[VEC ? MT : 1][4], xhv[VEC ? MT : 1][4];
            if constexpr (VEC) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < ntok) {
                        ld4(xt.tile(m) + TL::D + 16 * hf, xdv[m]);
                        ld4(xt.tile(m) + TL::H + 16 * hf, xhv[m]);
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                uint32_t lw[2][8];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t(&w)[WW] = r ? w1 : w0;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        lw[r][k] = prmt(w[16 * hf + 8 * s + k], w[16 * hf + 8 * s + k + 1], sel[r]);
                }
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int t = s + 2 * tt, u = 4 * hf + t;
                    uint32_t c[2][8];
                    int sA[2], sB[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            c[r][k] = ((lw[r][k] >> (4 * tt)) & 0x0f0f0f0fu) | (((hw[r][k] >> (2 * t)) & 0x03030303u) << 4);
                        const uint32_t scw = t < 2 ? scA[r] : scB[r];
                        sA[r] = (int)(int8_t)((scw >> (16 * (t & 1))) & 255u);
                        sB[r] = (int)(int8_t)((scw >> (16 * (t & 1) + 8)) & 255u);
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < ntok) {
                            const SAddr tl = xt.tile(m);
                            uint32_t x[8];
                            ldx8(tl + 32 * u, x);
                            const uint32_t xh = VEC ? xhv[VEC ? m : 0][t] : lds32(tl + TL::H + 4 * u);
                            const float xd = VEC ? __uint_as_float(xdv[VEC ? m : 0][t]) : ldsf(tl + TL::D + 4 * u);
                            const int hlo = (int)(int16_t)(xh & 0xffffu), hhi = (int)(int16_t)(xh >> 16);
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                int lo = 0, hi = 0;
#pragma unroll
                                for (int k = 0; k < 4; ++k) lo = dp4a(c[r][k], x[k], lo);
#pragma unroll
                                for (int k = 4; k < 8; ++k) hi = dp4a(c[r][k], x[k], hi);
                                const int dot = sA[r] * (lo - 32 * hlo) + sB[r] * (hi - 32 * hhi);
                                A[r][m] = fmaf(xd, (float)dot, A[r][m]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint32_t(&w)[WW] = r ? w1 : w0;
            const float d = half_bits_to_float(w[52] >> (8 * (r ? a1 : a0)));
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < ntok) sink.add(r, m, d * A[r][m]);
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void run(SAddr addr, int hf, const XT &xt, int ntok, Sink &sink) {
        uint32_t w[WW];
        load(addr, w);
        compute(w, (uint32_t)((uintptr_t)addr & 3u), hf, xt, ntok, sink);
    }
};

// ================================================================================ IQ4_XS
// T superblocks per task (136 bytes each; a two-superblock task is 16-byte aligned, a
// single one 8-byte aligned).  Value path: per token, sum_ib xd_ib * ((ls_ib - 32) *
// dot_ib), times d once per superblock.
template <int T>
struct FmtIQ4XS {
    static constexpr int QK = 256, BS = 136, XGT = 8 * T, TPB = 1, BPT = T, TASK_BYTES = 136 * T;
    static constexpr int WW = 34 * T;

    __device__ __forceinline__ static void load(SAddr addr, uint32_t (&w)[WW]) {
        if constexpr (T == 2) {
#pragma unroll
            for (int c = 0; c < WW / 4; ++c) {
                const uint4 v = lds128(addr + 16 * c);
                w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < WW / 2; ++c) {
                const uint2 v = lds64(addr + 8 * c);
                w[2 * c] = v.x;
                w[2 * c + 1] = v.y;
            }
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void superblock(const uint32_t *w, int u0, const XT &xt, int ntok,
                                                      Sink &sink) {
        using TL = Tile<XGT>;
        constexpr int MT = Sink::MT;
        const uint32_t h0 = w[0], h1 = w[1];  // h0: d | scales_h << 16, h1: scales_l[0..3]
        float A[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) A[m] = 0.0f;
        // up to 4 tokens: the 8 units' activation d of every token in two 16-byte loads
        // (more tokens: one 32-bit load per unit, to spare registers)
        constexpr bool VEC = MT <= 4;
        uint32_t xdv[VEC ? MT : 1][8];
        if constexpr (VEC && !Sink::DOTS) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < ntok) {
                    ld4(xt.tile(m) + TL::D + 4 * u0, xdv[m]);
                    ld4(xt.tile(m) + TL::D + 4 * u0 + 16, xdv[m] + 4);
                }
            }
        }
#pragma unroll
        for (int ib = 0; ib < 8; ++ib) {
            const int ls = (int)(((h1 >> (4 * ib)) & 15u) | (((h0 >> (16 + 2 * ib)) & 3u) << 4));
            uint32_t c[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) cb_lookup8(w[2 + 4 * ib + k], c[k], c[4 + k]);
            const int u = u0 + ib;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < ntok) {
                    const SAddr t = xt.tile(m);
                    uint32_t x[8];
                    ldx8(t + 32 * u, x);
                    int dot = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) dot = dp4a(c[k], x[k], dot);
                    if constexpr (Sink::DOTS) {
                        sink.unit(m, u, dot, 0);
                    } else {
                        const float xd = VEC ? __uint_as_float(xdv[VEC ? m : 0][ib]) : ldsf(t + TL::D + 4 * u);
                        A[m] = fmaf(xd, (float)((ls - 32) * dot), A[m]);
                    }
                }
            }
        }
        if constexpr (!Sink::DOTS) {
            const float d = half_bits_to_float(h0);
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < ntok) sink.add(m, d * A[m]);
        }
    }

    // Two rows' superblocks of the same column (T == 1) against the same activation tile;
    // per row the arithmetic and its order are superblock()'s.
    template <class PSink>
    __device__ __forceinline__ static void compute_pair(const uint32_t (&w0)[WW], uint32_t, const uint32_t (&w1)[WW],
                                                        uint32_t, const XT &xt, int ntok, PSink &sink) {
        static_assert(T == 1, "row pairs take one-superblock tasks");
        using TL = Tile<XGT>;
        constexpr int MT = PSink::MT;
        float A[2][MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) A[0][m] = A[1][m] = 0.0f;
        constexpr bool VEC = MT <= 4;
        uint32_t xdv[VEC ? MT : 1][8];
        if constexpr (VEC) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < ntok) {
                    ld4(xt.tile(m) + TL::D, xdv[m]);
                    ld4(xt.tile(m) + TL::D + 16, xdv[m] + 4);
                }
            }
        }
#pragma unroll
        for (int ib = 0; ib < 8; ++ib) {
            int ls[2];
            uint32_t c[2][8];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t(&w)[WW] = r ? w1 : w0;
                ls[r] = (int)(((w[1] >> (4 * ib)) & 15u) | (((w[0] >> (16 + 2 * ib)) & 3u) << 4));
#pragma unroll
                for (int k = 0; k < 4; ++k) cb_lookup8(w[2 + 4 * ib + k], c[r][k], c[r][4 + k]);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < ntok) {
                    const SAddr t = xt.tile(m);
                    uint32_t x[8];
                    ldx8(t + 32 * ib, x);
                    const float xd = VEC ? __uint_as_float(xdv[VEC ? m : 0][ib]) : ldsf(t + TL::D + 4 * ib);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        int dot = 0;
#pragma unroll
                        for (int k = 0; k < 8; ++k) dot = dp4a(c[r][k], x[k], dot);
                        A[r][m] = fmaf(xd, (float)((ls[r] - 32) * dot), A[r][m]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float d = half_bits_to_float((r ? w1 : w0)[0]);
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < ntok) sink.add(r, m, d * A[r][m]);
        }
    }

    template <class Sink>
    __device__ __forceinline__ static void compute(const uint32_t (&w)[WW], uint32_t, int, const XT &xt, int ntok,
                                                   Sink &sink) {
#pragma unroll
        for (int t = 0; t < T; ++t) superblock(w + 34 * t, 8 * t, xt, ntok, sink);
    }

    template <class Sink>
    __device__ __forceinline__ static void run(SAddr addr, int hf, const XT &xt, int ntok, Sink &sink) {
        uint32_t w[WW];
        load(addr, w);
        compute(w, 0, hf, xt, ntok, sink);
    }
};

// ================================================================================ selection
template <int FMT, int T>
struct FmtSel;
template <int T>
struct FmtSel<F_Q8_0, T> { using type = FmtLegacy<F_Q8_0, T>; };
template <int T>
struct FmtSel<F_Q4_0, T> { using type = FmtLegacy<F_Q4_0, T>; };
template <int T>
struct FmtSel<F_Q4_1, T> { using type = FmtLegacy<F_Q4_1, T>; };
template <int T>
struct FmtSel<F_Q5_0, T> { using type = FmtLegacy<F_Q5_0, T>; };
template <int T>
struct FmtSel<F_Q5_1, T> { using type = FmtLegacy<F_Q5_1, T>; };
template <int T>
struct FmtSel<F_IQ4_NL, T> { using type = FmtLegacy<F_IQ4_NL, T>; };
template <int T>
struct FmtSel<F_Q2_K, T> { using type = FmtQ2K<T>; };
template <int T>
struct FmtSel<F_Q3_K, T> { using type = FmtQ3K<T>; };
template <int T>
struct FmtSel<F_Q4_K, T> { using type = FmtQ4K<T>; };
template <int T>
struct FmtSel<F_Q5_K, T> { using type = FmtQ5K<T>; };
template <int T>
struct FmtSel<F_Q6_K, T> { using type = FmtQ6K<T>; };
template <int T>
struct FmtSel<F_IQ4_XS, T> { using type = FmtIQ4XS<T>; };
template <int FMT, int T>
using FT = typename FmtSel<FMT, T>::type;

// ================================================================================ tile writer
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// One activation block (lane i holds code i) into unit u of a task tile of xgt units:
// codes, then per unit d, s, the two 16-element half sums packed in 16 bits each, d * s.
__device__ __forceinline__ void put_tile_unit(uint8_t *t, int u, int xgt, int lane, int qi, float di, int si) {
    t[32 * u + lane] = (uint8_t)qi;
    const int h16 = __reduce_add_sync(0xffffffffu, lane < 16 ? qi : 0);
    if (lane == 0) {
        reinterpret_cast<float *>(t + 32 * xgt)[u] = di;
        reinterpret_cast<int32_t *>(t + 36 * xgt)[u] = si;
        reinterpret_cast<uint32_t *>(t + 40 * xgt)[u] = ((uint32_t)h16 & 0xffffu) | ((uint32_t)(si - h16) << 16);
        reinterpret_cast<float *>(t + 44 * xgt)[u] = di * (float)si;
    }
}

// Quantized activation block b (32 codes, one per lane) of image row r, in an image of tpr
// tasks per row of 2^xgt_log2 blocks each.
__device__ __forceinline__ void put_block(uint8_t *img, long r, int tpr, int b, int xgt_log2, int lane, int q,
                                          float d, int s) {
    const int xgt = 1 << xgt_log2;
    put_tile_unit(img + (r * tpr + (b >> xgt_log2)) * tile_stride(xgt), b & (xgt - 1), xgt, lane, q, d, s);
}

// An s16 block of activation row r as its two int8 planes (see prep_tiles_s16_warp): image
// rows 2r (hi, step 256 d) and 2r + 1 (lo, step d).
__device__ __forceinline__ void put_block_s16(uint8_t *img, long r, int tpr, int b, int xgt_log2, int lane, int q,
                                              float d, int s) {
    const int hi = (q + 128) >> 8, lo = q - 256 * hi;
    const int shi = __reduce_add_sync(0xffffffffu, hi);
    put_block(img, 2 * r, tpr, b, xgt_log2, lane, hi, 256.0f * d, shi);
    put_block(img, 2 * r + 1, tpr, b, xgt_log2, lane, lo, d, s - 256 * shi);
}

// Activation rows -> task-tile image in global memory: tile (row r, task tt) at
// img + (r * tpr + tt) * tile_stride(xgt).  One warp per activation block; lane i holds
// element i.  src_f32 != nullptr: quantize fp32 rows (activation quantization rule) --
// with u != nullptr the rows are h = silu(src_f32) * u (SwiGLU), also stored to h_out when
// given -- else repack already-quantized rows (q: row pitch K; d/s: row pitch K/32).
// mq/md/ms (nullable): the quantized rows in their plain layout as well.
__device__ __forceinline__ void prep_tiles_warp(const float *src_f32, const float *u, float *h_out, const int8_t *q,
                                                const float *d, const int32_t *s, int rows, int K, int xgt_log2,
                                                uint8_t *img, int8_t *mq, float *md, int32_t *ms, long wid,
                                                long nwarps) {
    const int lane = threadIdx.x & 31;
    const int nb = K / 32, tpr = nb >> xgt_log2;
    for (long w = wid; w < (long)rows * nb; w += nwarps) {
        const int r = (int)(w / nb), b = (int)(w - (long)r * nb);
        int qi, si;
        float di;
        if (src_f32) {
            const long idx = (long)r * K + 32L * b + lane;
            float v = src_f32[idx];
            if (u) {
                v = silu_mul(v, u[idx]);
                if (h_out) h_out[idx] = v;
            }
            quant_block_warp(v, qi, di, si);
        } else {
            qi = q[(long)r * K + 32L * b + lane];
            di = d[(long)r * nb + b];
            si = s[(long)r * nb + b];
        }
        put_block(img, r, tpr, b, xgt_log2, lane, qi, di, si);
        if (mq) {
            mq[(long)r * K + 32L * b + lane] = (int8_t)qi;
            if (lane == 0) {
                md[(long)r * nb + b] = di;
                ms[(long)r * nb + b] = si;
            }
        }
    }
}

// s16 activation rows -> task-tile image of two int8 planes per row.  An s16 code q is
// split as q = 256 * hi + lo with hi = (q + 128) >> 8 in [-127, 127] and lo in [-128, 127];
// image row 2r holds the hi plane with step 256 * d (exact: a power-of-two scaling), row
// 2r + 1 the lo plane with step d, each in the int8 tile layout (put_block_s16).  Every
// per-unit term the engines form from a row (d * dot, d * s, the min-code sums) is linear
// in the codes, so the two planes' results add up to the s16 result with the exact integer
// sums.  One warp per activation block of the fp32 rows x.
__device__ __forceinline__ void prep_tiles_s16_warp(const float *x, int rows, int K, int xgt_log2, uint8_t *img,
                                                    long wid, long nwarps) {
    const int lane = threadIdx.x & 31;
    const int nb = K / 32, tpr = nb >> xgt_log2;
    for (long w = wid; w < (long)rows * nb; w += nwarps) {
        const int r = (int)(w / nb), b = (int)(w - (long)r * nb);
        int q, s;
        float d;
        quant_block_warp16(x[(long)r * K + 32L * b + lane], q, d, s);
        put_block_s16(img, r, tpr, b, xgt_log2, lane, q, d, s);
    }
}

}  // namespace qg
