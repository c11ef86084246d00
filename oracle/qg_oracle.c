/*
 * qg_oracle.c -- plain CPU oracle (TEST INFRASTRUCTURE ONLY; see qg_oracle.h).
 *
 * Written for a reader to check by eye against the definitions: one element at a
 * time, no blocking, no SIMD, fp64 throughout except where the method fixes fp32.
 * The only parallelism is an OpenMP loop over independent output rows, which does
 * not change any result.
 */
#include "qg_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 0; /* 0: OpenMP default */

void or_set_threads(int n) { g_threads = n; }

int or_get_threads(void) {
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

int or_block_elems(int fmt) {
    switch (fmt) {
    case OR_Q4_0: case OR_Q4_1: case OR_Q5_0: case OR_Q5_1: case OR_Q8_0: case OR_IQ4_NL: return 32;
    case OR_Q2_K: case OR_Q3_K: case OR_Q4_K: case OR_Q5_K: case OR_Q6_K: case OR_IQ4_XS: return 256;
    default: return 0;
    }
}

int or_block_bytes(int fmt) {
    switch (fmt) {
    case OR_Q4_0: return 18;    /* fp16 d + 16 bytes of nibbles              */
    case OR_Q4_1: return 20;    /* fp16 d, fp16 m + 16 bytes of nibbles      */
    case OR_Q5_0: return 22;    /* fp16 d, 32 fifth bits, 16 B of nibbles     */
    case OR_Q5_1: return 24;    /* fp16 d, fp16 m, 32 fifth bits, nibbles     */
    case OR_IQ4_NL: return 18;  /* fp16 d + 16 bytes of codebook indices      */
    case OR_Q8_0: return 34;    /* fp16 d + 32 int8                          */
    case OR_Q2_K: return 84;    /* 16 B 4-bit scale|min, 64 B 2-bit codes, d, dmin */
    case OR_Q3_K: return 110;   /* 32 B high bits, 64 B 2-bit codes, 12 B scales, d */
    case OR_Q4_K: return 144;   /* d, dmin, 12 B scales/mins, 128 B nibbles   */
    case OR_Q5_K: return 176;   /* Q4_K fields + 32 B of fifth bits           */
    case OR_Q6_K: return 210;   /* 128 B ql, 64 B qh, 16 int8 scales, fp16 d  */
    case OR_IQ4_XS: return 136; /* d, u16 scales_h, 4 B scales_l, 128 B index */
    default: return 0;
    }
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double or_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static double rd_half(const uint8_t *p) { return or_half_to_double(rd_u16(p)); }

/* The 16-entry non-linear codebook of IQ4_NL / IQ4_XS (public GGUF definition;
 * the page speaks only of "a tiny codebook kept in registers"). */
static const int8_t kIQ4NL[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                  1,    13,   25,  38,  53,  69,  89,  113};

/* Q4_K / Q5_K: 6-bit scale S_j and min M_j of sub-block j (0..7) packed in 12 bytes. */
static void kquant_scale_min(const uint8_t *sc12, int j, int *S, int *M) {
    if (j < 4) {
        *S = sc12[j] & 63;
        *M = sc12[j + 4] & 63;
    } else {
        *S = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
        *M = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
    }
}

/* Q3_K: the signed 6-bit scale of 16-element sub-block i (0..15), packed in 12 bytes:
 * its low 4 bits are the low nibble of byte i (i < 8) or the high nibble of byte i-8,
 * its high 2 bits are bits 2*(i/4), 2*(i/4)+1 of byte 8 + i%4; the value is that - 32. */
static int q3k_scale(const uint8_t *sc12, int i) {
    int low4 = i < 8 ? (sc12[i] & 15) : (sc12[i - 8] >> 4);
    int high2 = (sc12[8 + i % 4] >> (2 * (i / 4))) & 3;
    return (low4 | (high2 << 4)) - 32;
}

void or_decode_block(int fmt, const uint8_t *blk, double *w, int32_t *c, double *A, double *B) {
    or_decode_block_mc(fmt, blk, w, c, NULL, A, B);
}

void or_decode_block_mc(int fmt, const uint8_t *blk, double *w, int32_t *c, int32_t *mc, double *A, double *B) {
    int QK = or_block_elems(fmt);
    for (int e = 0; e < QK; ++e) {
        int u = e / 32;        /* 32-element unit (= one activation block) */
        int code = 0;          /* contract code c_e                        */
        int mcode = 1;         /* min code mc_e                            */
        double a = 0, b = 0;   /* w_e = a * c_e - b * mc_e                 */
        switch (fmt) {
        case OR_Q8_0: {
            a = rd_half(blk);
            code = (int8_t)blk[2 + e];
            break;
        }
        case OR_Q4_0: {
            a = rd_half(blk);
            int nib = e < 16 ? (blk[2 + e] & 15) : (blk[2 + e - 16] >> 4);
            code = nib - 8;
            break;
        }
        case OR_Q4_1: {
            /* fp16 d, fp16 m, nibbles as Q4_0; w = d * nibble + m */
            a = rd_half(blk);
            b = -rd_half(blk + 2);
            code = e < 16 ? (blk[4 + e] & 15) : (blk[4 + e - 16] >> 4);
            break;
        }
        case OR_Q5_0:
        case OR_Q5_1: {
            /* fp16 d, [fp16 m,] 32-bit little-endian qh (bit e = fifth bit of element e),
             * nibbles as Q4_0; Q5_0: w = d * (code - 16), Q5_1: w = d * code + m */
            const int one = fmt == OR_Q5_1;
            a = rd_half(blk);
            const uint8_t *qh = blk + (one ? 4 : 2), *qs = blk + (one ? 8 : 6);
            int nib = e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);
            int hb = (qh[e / 8] >> (e % 8)) & 1;
            code = nib | (hb << 4);
            if (one) b = -rd_half(blk + 2);
            else code -= 16;
            break;
        }
        case OR_IQ4_NL: {
            /* fp16 d, 16 bytes of 4-bit codebook indices laid out as Q4_0 nibbles */
            a = rd_half(blk);
            int idx = e < 16 ? (blk[2 + e] & 15) : (blk[2 + e - 16] >> 4);
            code = kIQ4NL[idx];
            break;
        }
        case OR_Q4_K:
        case OR_Q5_K: {
            double d = rd_half(blk), dmin = rd_half(blk + 2);
            const uint8_t *sc12 = blk + 4;
            const uint8_t *qh = blk + 16;                       /* Q5_K only */
            const uint8_t *qs = blk + (fmt == OR_Q4_K ? 16 : 48);
            int j = e / 32, l = e % 32, S, M;
            kquant_scale_min(sc12, j, &S, &M);
            int byte = qs[32 * (j / 2) + l];
            int nib = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
            if (fmt == OR_Q5_K) nib += 16 * ((qh[l] >> j) & 1);
            code = nib;
            a = d * S;
            b = dmin * M;
            break;
        }
        case OR_Q2_K:
        case OR_Q3_K: {
            /* Element e = 128h + 32j + l: its 2-bit code is bits 2j, 2j+1 of qs[32h + l];
             * it belongs to 16-element sub-block e/16.
             * Q2_K: scales[16] @0 (low nibble: scale, high nibble: min), qs @16, fp16 d @80,
             *       fp16 dmin @82; w = d * scale * code - dmin * min.
             * Q3_K: hmask[32] @0, qs @32, 12 B packed scales @96, fp16 d @108; the third bit of
             *       the code is bit 4h + j of hmask[l], and a clear bit subtracts 4:
             *       w = d * (scale - 32) * (code - 4 * (1 - bit)). */
            int h = e / 128, r = e % 128, j = r / 32, l = r % 32, sb = e / 16;
            if (fmt == OR_Q2_K) {
                int q2 = (blk[16 + 32 * h + l] >> (2 * j)) & 3;
                code = (blk[sb] & 15) * q2;
                mcode = blk[sb] >> 4;
                a = rd_half(blk + 80);
                b = rd_half(blk + 82);
            } else {
                int q2 = (blk[32 + 32 * h + l] >> (2 * j)) & 3;
                int hb = (blk[l] >> (4 * h + j)) & 1;
                code = q3k_scale(blk + 96, sb) * (q2 - (hb ? 0 : 4));
                a = rd_half(blk + 108);
            }
            break;
        }
        case OR_Q6_K: {
            const uint8_t *ql = blk, *qh = blk + 128;
            const int8_t *sc = (const int8_t *)(blk + 192);
            double d = rd_half(blk + 208);
            int h = e / 128, r = e % 128, l = r % 32, t = r / 32;
            int lbyte = ql[64 * h + l + 32 * (t & 1)];
            int low4 = (t < 2) ? (lbyte & 15) : (lbyte >> 4);
            int hi2 = (qh[32 * h + l] >> (2 * t)) & 3;
            int q6 = low4 | (hi2 << 4);
            code = sc[e / 16] * (q6 - 32);
            a = d;
            break;
        }
        case OR_IQ4_XS: {
            double d = rd_half(blk);
            int scales_h = rd_u16(blk + 2);
            const uint8_t *scales_l = blk + 4, *qs = blk + 8;
            int ib = e / 32, j = e % 32;
            int ls = ((scales_l[ib / 2] >> (4 * (ib % 2))) & 15) | (((scales_h >> (2 * ib)) & 3) << 4);
            int byte = qs[16 * ib + (j % 16)];
            int idx = (j < 16) ? (byte & 15) : (byte >> 4);
            code = kIQ4NL[idx];
            a = d * (ls - 32);
            break;
        }
        default:
            return;
        }
        if (w) w[e] = a * code - b * mcode;
        if (c) c[e] = code;
        if (mc) mc[e] = mcode;
        if (e % 32 == 0) {
            if (A) A[u] = a;
            if (B) B[u] = b;
        }
    }
}

void or_dequant_matrix(int fmt, const uint8_t *W, int N, int K, double *out) {
    int QK = or_block_elems(fmt), BS = or_block_bytes(fmt), nb = K / QK;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b)
            or_decode_block(fmt, W + ((size_t)n * nb + b) * BS, out + (size_t)n * K + (size_t)b * QK,
                            NULL, NULL, NULL);
}

/* Activation codes of either width: exactly one of q8, q16 is non-NULL. */
typedef struct {
    const int8_t *q8;
    const int16_t *q16;
} or_codes;

static int32_t code_at(or_codes a, size_t i) { return a.q8 ? (int32_t)a.q8[i] : (int32_t)a.q16[i]; }

/* Activation quantization, one 32-element block at a time, to codes in [-qmax, qmax]
 * with d = amax / qmax.  The page names the int8 activation format "Q8_F32S" only; the
 * per-32 block, the fp32 scale, round half away from zero and true division are the
 * readings taken here.  q8 or q16 receives the codes. */
static void quantize_rows(const float *x, int M, int K, float qmax, int8_t *q8, int16_t *q16, float *xd,
                          int32_t *xs) {
    int nb = K / 32, lim = (int)qmax;
    for (int m = 0; m < M; ++m) {
        for (int b = 0; b < nb; ++b) {
            const float *xb = x + (size_t)m * K + (size_t)b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / qmax;                  /* fp32, round to nearest even */
            int32_t s = 0;
            for (int i = 0; i < 32; ++i) {
                int q = 0;
                if (d != 0.0f) {
                    float v = xb[i] / d;            /* fp32 IEEE division */
                    q = (int)roundf(v);             /* half away from zero */
                    if (q > lim) q = lim;
                    if (q < -lim) q = -lim;
                }
                size_t o = (size_t)m * K + (size_t)b * 32 + i;
                if (q8) q8[o] = (int8_t)q;
                else q16[o] = (int16_t)q;
                s += q;
            }
            xd[(size_t)m * nb + b] = d;
            xs[(size_t)m * nb + b] = s;
        }
    }
}

void or_quantize_act(const float *x, int M, int K, int8_t *xq, float *xd, int32_t *xs) {
    quantize_rows(x, M, K, 127.0f, xq, NULL, xd, xs);
}

/* s16 activations ([KES] section 四, issue ⑫: the MoE FFN moved from int8 to s16
 * activations, the quantization step 256 times finer).  Reading: the step is the int8
 * step divided by 256, d = amax / (127 * 256) = amax / 32512 (in fp32 the same as
 * (amax / 127) / 256: a power-of-two scaling), and the codes lie in [-32512, 32512]. */
void or_quantize_act16(const float *x, int M, int K, int16_t *xq, float *xd, int32_t *xs) {
    quantize_rows(x, M, K, 32512.0f, NULL, xq, xd, xs);
}

static int has_min_term(int fmt) {
    return fmt == OR_Q4_K || fmt == OR_Q5_K || fmt == OR_Q4_1 || fmt == OR_Q5_1 || fmt == OR_Q2_K;
}

void or_block_dots(int fmt, const uint8_t *W, const int8_t *xq, const int32_t *xs,
                   int N, int K, int M, int32_t *dots, int32_t *aux) {
    int QK = or_block_elems(fmt), BS = or_block_bytes(fmt), nb = K / QK, nu = K / 32;
    int upb = QK / 32;
#pragma omp parallel for schedule(static) num_threads(or_get_threads())
    for (int n = 0; n < N; ++n) {
        int32_t c[256], mc[256];
        for (int b = 0; b < nb; ++b) {
            or_decode_block_mc(fmt, W + ((size_t)n * nb + b) * BS, NULL, c, mc, NULL, NULL);
            for (int ub = 0; ub < upb; ++ub) {
                int u = b * upb + ub;
                for (int m = 0; m < M; ++m) {
                    const int8_t *q = xq + (size_t)m * K + (size_t)u * 32;
                    int32_t dot = 0, msum = 0;
                    for (int i = 0; i < 32; ++i) {
                        dot += c[ub * 32 + i] * (int32_t)q[i];
                        msum += mc[ub * 32 + i] * (int32_t)q[i];
                    }
                    size_t o = ((size_t)m * N + n) * nu + u;
                    dots[o] = dot;
                    if (aux) {
                        /* the per-16 mins of Q2_K enter through their own sum; for the
                         * other formats mc = 1 and the sum is the activation sum xs */
                        int32_t a = fmt == OR_Q2_K ? msum : xs[(size_t)m * nu + u];
                        aux[o] = has_min_term(fmt) ? a : 0;
                    }
                }
            }
        }
    }
}

static void gemv_codes(int fmt, const uint8_t *W, or_codes xq, const float *xd, const int32_t *xs,
                       int N, int K, int M, double *y) {
    int QK = or_block_elems(fmt), BS = or_block_bytes(fmt), nb = K / QK, nu = K / 32;
    int upb = QK / 32;
#pragma omp parallel for schedule(static) num_threads(or_get_threads())
    for (int n = 0; n < N; ++n) {
        int32_t c[256], mc[256];
        double A[8], B[8];
        for (int m = 0; m < M; ++m) y[(size_t)m * N + n] = 0.0;
        for (int b = 0; b < nb; ++b) {
            or_decode_block_mc(fmt, W + ((size_t)n * nb + b) * BS, NULL, c, mc, A, B);
            for (int ub = 0; ub < upb; ++ub) {
                int u = b * upb + ub;
                for (int m = 0; m < M; ++m) {
                    size_t q0 = (size_t)m * K + (size_t)u * 32;
                    int32_t dot = 0, msum = 0;
                    for (int i = 0; i < 32; ++i) {
                        dot += c[ub * 32 + i] * code_at(xq, q0 + i);
                        msum += mc[ub * 32 + i] * code_at(xq, q0 + i);
                    }
                    double d_x = xd[(size_t)m * nu + u];
                    double s_x = fmt == OR_Q2_K ? (double)msum : (double)xs[(size_t)m * nu + u];
                    y[(size_t)m * N + n] += d_x * (A[ub] * (double)dot - B[ub] * s_x);
                }
            }
        }
    }
}

void or_gemv_q(int fmt, const uint8_t *W, const int8_t *xq, const float *xd, const int32_t *xs,
               int N, int K, int M, double *y) {
    or_codes a = {xq, NULL};
    gemv_codes(fmt, W, a, xd, xs, N, K, M, y);
}

void or_gemv_q16(int fmt, const uint8_t *W, const int16_t *xq, const float *xd, const int32_t *xs,
                 int N, int K, int M, double *y) {
    or_codes a = {NULL, xq};
    gemv_codes(fmt, W, a, xd, xs, N, K, M, y);
}

void or_gemv_deq(int fmt, const uint8_t *W, const int8_t *xq, const float *xd,
                 int N, int K, int M, double *y) {
    int QK = or_block_elems(fmt), BS = or_block_bytes(fmt), nb = K / QK, nu = K / 32;
#pragma omp parallel for schedule(static) num_threads(or_get_threads())
    for (int n = 0; n < N; ++n) {
        double w[256];
        for (int m = 0; m < M; ++m) y[(size_t)m * N + n] = 0.0;
        for (int b = 0; b < nb; ++b) {
            or_decode_block(fmt, W + ((size_t)n * nb + b) * BS, w, NULL, NULL, NULL);
            for (int e = 0; e < QK; ++e) {
                int k = b * QK + e;
                for (int m = 0; m < M; ++m) {
                    double xhat = (double)xq[(size_t)m * K + k] * (double)xd[(size_t)m * nu + k / 32];
                    y[(size_t)m * N + n] += w[e] * xhat;
                }
            }
        }
    }
}

static void absdot_codes(int fmt, const uint8_t *W, or_codes xq, const float *xd,
                         int N, int K, int M, double *sabs) {
    int QK = or_block_elems(fmt), BS = or_block_bytes(fmt), nb = K / QK, nu = K / 32;
#pragma omp parallel for schedule(static) num_threads(or_get_threads())
    for (int n = 0; n < N; ++n) {
        double w[256];
        for (int m = 0; m < M; ++m) sabs[(size_t)m * N + n] = 0.0;
        for (int b = 0; b < nb; ++b) {
            or_decode_block(fmt, W + ((size_t)n * nb + b) * BS, w, NULL, NULL, NULL);
            for (int e = 0; e < QK; ++e) {
                int k = b * QK + e;
                for (int m = 0; m < M; ++m) {
                    double xhat = (double)code_at(xq, (size_t)m * K + k) * (double)xd[(size_t)m * nu + k / 32];
                    sabs[(size_t)m * N + n] += fabs(w[e] * xhat);
                }
            }
        }
    }
}

void or_absdot(int fmt, const uint8_t *W, const int8_t *xq, const float *xd,
               int N, int K, int M, double *sabs) {
    or_codes a = {xq, NULL};
    absdot_codes(fmt, W, a, xd, N, K, M, sabs);
}

void or_absdot16(int fmt, const uint8_t *W, const int16_t *xq, const float *xd,
                 int N, int K, int M, double *sabs) {
    or_codes a = {NULL, xq};
    absdot_codes(fmt, W, a, xd, N, K, M, sabs);
}

void or_gemv(int fmt, const uint8_t *W, const float *x, int N, int K, int M, double *y) {
    int8_t *xq = (int8_t *)malloc((size_t)M * K);
    float *xd = (float *)malloc(sizeof(float) * (size_t)M * (K / 32));
    int32_t *xs = (int32_t *)malloc(sizeof(int32_t) * (size_t)M * (K / 32));
    or_quantize_act(x, M, K, xq, xd, xs);
    or_gemv_q(fmt, W, xq, xd, xs, N, K, M, y);
    free(xq);
    free(xd);
    free(xs);
}

void or_router(const float *x, int M, int H, const float *Wr, int E, int topk,
               double *logits, double *probs, int32_t *ids, double *w) {
    double *l = (double *)malloc(sizeof(double) * E);
    double *p = (double *)malloc(sizeof(double) * E);
    char *taken = (char *)malloc(E);
    for (int m = 0; m < M; ++m) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int k = 0; k < H; ++k) acc += (double)Wr[(size_t)e * H + k] * (double)x[(size_t)m * H + k];
            l[e] = acc;
        }
        double lmax = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > lmax) lmax = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - lmax); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= z;
        if (logits) for (int e = 0; e < E; ++e) logits[(size_t)m * E + e] = l[e];
        if (probs) for (int e = 0; e < E; ++e) probs[(size_t)m * E + e] = p[e];
        /* top-k by repeated selection of the largest remaining probability; a tie
         * keeps the lower expert id because only a strictly larger value replaces it */
        memset(taken, 0, E);
        double wsum = 0.0;
        for (int s = 0; s < topk; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
            taken[best] = 1;
            ids[(size_t)m * topk + s] = best;
            w[(size_t)m * topk + s] = p[best];
            wsum += p[best];
        }
        for (int s = 0; s < topk; ++s) w[(size_t)m * topk + s] /= wsum;
    }
    free(l);
    free(p);
    free(taken);
}

double or_swiglu(double g, double u) { return g * u / (1.0 + exp(-g)); }

static size_t matrix_bytes(int fmt, int rows, int cols) {
    return (size_t)rows * (size_t)(cols / or_block_elems(fmt)) * (size_t)or_block_bytes(fmt);
}

/* The MoE stages take the activation width as a parameter: bits = 8 (the int8 rule) or
 * 16 (the s16 rule); codes of the other width are never formed. */
static void moe_gateup_bits(int bits, int fmt, const float *x, int M, int H, int E, int topk, int I,
                            const int32_t *ids, const uint8_t *Wg_exps, const uint8_t *Wu_exps,
                            const uint8_t *Wg_sh, const uint8_t *Wu_sh,
                            double *g, double *u, double *h) {
    (void)E;
    int S = topk + 1;
    size_t eb = matrix_bytes(fmt, I, H);
    int8_t *q8 = bits == 8 ? (int8_t *)malloc((size_t)H) : NULL;
    int16_t *q16 = bits == 16 ? (int16_t *)malloc(sizeof(int16_t) * (size_t)H) : NULL;
    or_codes xq = {q8, q16};
    float *xd = (float *)malloc(sizeof(float) * (H / 32));
    int32_t *xs = (int32_t *)malloc(sizeof(int32_t) * (H / 32));
    double *gg = (double *)malloc(sizeof(double) * I);
    double *uu = (double *)malloc(sizeof(double) * I);
    for (int m = 0; m < M; ++m) {
        /* x quantized once per token */
        quantize_rows(x + (size_t)m * H, 1, H, bits == 8 ? 127.0f : 32512.0f, q8, q16, xd, xs);
        for (int s = 0; s < S; ++s) {
            const uint8_t *Wg = s < topk ? Wg_exps + eb * (size_t)ids[(size_t)m * topk + s] : Wg_sh;
            const uint8_t *Wu = s < topk ? Wu_exps + eb * (size_t)ids[(size_t)m * topk + s] : Wu_sh;
            gemv_codes(fmt, Wg, xq, xd, xs, I, H, 1, gg);
            gemv_codes(fmt, Wu, xq, xd, xs, I, H, 1, uu);
            for (int j = 0; j < I; ++j) {
                size_t o = ((size_t)m * S + s) * I + j;
                if (g) g[o] = gg[j];
                if (u) u[o] = uu[j];
                if (h) h[o] = or_swiglu(gg[j], uu[j]);
            }
        }
    }
    free(q8); free(q16); free(xd); free(xs); free(gg); free(uu);
}

void or_moe_gateup(int fmt, const float *x, int M, int H, int E, int topk, int I,
                   const int32_t *ids, const uint8_t *Wg_exps, const uint8_t *Wu_exps,
                   const uint8_t *Wg_sh, const uint8_t *Wu_sh,
                   double *g, double *u, double *h) {
    moe_gateup_bits(8, fmt, x, M, H, E, topk, I, ids, Wg_exps, Wu_exps, Wg_sh, Wu_sh, g, u, h);
}

void or_moe_gateup16(int fmt, const float *x, int M, int H, int E, int topk, int I,
                     const int32_t *ids, const uint8_t *Wg_exps, const uint8_t *Wu_exps,
                     const uint8_t *Wg_sh, const uint8_t *Wu_sh,
                     double *g, double *u, double *h) {
    moe_gateup_bits(16, fmt, x, M, H, E, topk, I, ids, Wg_exps, Wu_exps, Wg_sh, Wu_sh, g, u, h);
}

static float *h_to_fp32(const double *h, size_t n) {
    float *hf = (float *)malloc(sizeof(float) * n);
    for (size_t i = 0; i < n; ++i) hf[i] = (float)h[i];   /* round to nearest fp32 */
    return hf;
}

void or_requant(const double *h, int R, int I, int8_t *hq, float *hd, int32_t *hs) {
    float *hf = h_to_fp32(h, (size_t)R * I);
    or_quantize_act(hf, R, I, hq, hd, hs);
    free(hf);
}

void or_requant16(const double *h, int R, int I, int16_t *hq, float *hd, int32_t *hs) {
    float *hf = h_to_fp32(h, (size_t)R * I);
    or_quantize_act16(hf, R, I, hq, hd, hs);
    free(hf);
}

static void moe_down_codes(int fmt, int M, int H, int E, int topk, int I,
                           const int32_t *ids, const double *w,
                           or_codes hq, const float *hd, const int32_t *hs,
                           const uint8_t *Wd_exps, const uint8_t *Wd_sh,
                           double *y, double *o, double *yabs) {
    (void)E;
    int S = topk + 1, nu = I / 32;
    size_t eb = matrix_bytes(fmt, H, I);
    double *oo = (double *)malloc(sizeof(double) * H);
    double *aa = (double *)malloc(sizeof(double) * H);
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < H; ++n) {
            y[(size_t)m * H + n] = 0.0;
            if (yabs) yabs[(size_t)m * H + n] = 0.0;
        }
        for (int s = 0; s < S; ++s) {
            const uint8_t *Wd = s < topk ? Wd_exps + eb * (size_t)ids[(size_t)m * topk + s] : Wd_sh;
            double ws = s < topk ? w[(size_t)m * topk + s] : 1.0;     /* shared expert: weight 1 */
            size_t r = (size_t)m * S + s;
            or_codes hr = {hq.q8 ? hq.q8 + r * I : NULL, hq.q16 ? hq.q16 + r * I : NULL};
            gemv_codes(fmt, Wd, hr, hd + r * nu, hs + r * nu, H, I, 1, oo);
            if (yabs) absdot_codes(fmt, Wd, hr, hd + r * nu, H, I, 1, aa);
            for (int n = 0; n < H; ++n) {
                y[(size_t)m * H + n] += ws * oo[n];
                if (o) o[r * H + n] = oo[n];
                if (yabs) yabs[(size_t)m * H + n] += fabs(ws) * aa[n];
            }
        }
    }
    free(oo);
    free(aa);
}

void or_moe_down(int fmt, int M, int H, int E, int topk, int I,
                 const int32_t *ids, const double *w,
                 const int8_t *hq, const float *hd, const int32_t *hs,
                 const uint8_t *Wd_exps, const uint8_t *Wd_sh,
                 double *y, double *o, double *yabs) {
    or_codes a = {hq, NULL};
    moe_down_codes(fmt, M, H, E, topk, I, ids, w, a, hd, hs, Wd_exps, Wd_sh, y, o, yabs);
}

void or_moe_down16(int fmt, int M, int H, int E, int topk, int I,
                   const int32_t *ids, const double *w,
                   const int16_t *hq, const float *hd, const int32_t *hs,
                   const uint8_t *Wd_exps, const uint8_t *Wd_sh,
                   double *y, double *o, double *yabs) {
    or_codes a = {NULL, hq};
    moe_down_codes(fmt, M, H, E, topk, I, ids, w, a, hd, hs, Wd_exps, Wd_sh, y, o, yabs);
}

static void moe_ffn_bits(int bits, int fmt, const float *x, int M, int H, const float *Wr, int E, int topk,
                         const uint8_t *Wg_exps, const uint8_t *Wu_exps, const uint8_t *Wd_exps,
                         const uint8_t *Wg_sh, const uint8_t *Wu_sh, const uint8_t *Wd_sh, int I,
                         double *y, int32_t *ids, double *w) {
    int S = topk + 1;
    size_t R = (size_t)M * S;
    or_router(x, M, H, Wr, E, topk, NULL, NULL, ids, w);
    double *h = (double *)malloc(sizeof(double) * R * I);
    int8_t *q8 = bits == 8 ? (int8_t *)malloc(R * I) : NULL;
    int16_t *q16 = bits == 16 ? (int16_t *)malloc(sizeof(int16_t) * R * I) : NULL;
    or_codes hq = {q8, q16};
    float *hd = (float *)malloc(sizeof(float) * R * (I / 32));
    int32_t *hs = (int32_t *)malloc(sizeof(int32_t) * R * (I / 32));
    moe_gateup_bits(bits, fmt, x, M, H, E, topk, I, ids, Wg_exps, Wu_exps, Wg_sh, Wu_sh, NULL, NULL, h);
    float *hf = h_to_fp32(h, R * I);
    quantize_rows(hf, (int)R, I, bits == 8 ? 127.0f : 32512.0f, q8, q16, hd, hs);
    moe_down_codes(fmt, M, H, E, topk, I, ids, w, hq, hd, hs, Wd_exps, Wd_sh, y, NULL, NULL);
    free(h); free(hf); free(q8); free(q16); free(hd); free(hs);
}

void or_moe_ffn(int fmt, const float *x, int M, int H, const float *Wr, int E, int topk,
                const uint8_t *Wg_exps, const uint8_t *Wu_exps, const uint8_t *Wd_exps,
                const uint8_t *Wg_sh, const uint8_t *Wu_sh, const uint8_t *Wd_sh, int I,
                double *y, int32_t *ids, double *w) {
    moe_ffn_bits(8, fmt, x, M, H, Wr, E, topk, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I, y, ids, w);
}

void or_moe_ffn16(int fmt, const float *x, int M, int H, const float *Wr, int E, int topk,
                  const uint8_t *Wg_exps, const uint8_t *Wu_exps, const uint8_t *Wd_exps,
                  const uint8_t *Wg_sh, const uint8_t *Wu_sh, const uint8_t *Wd_sh, int I,
                  double *y, int32_t *ids, double *w) {
    moe_ffn_bits(16, fmt, x, M, H, Wr, E, topk, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I, y, ids, w);
}

void or_ffn_sublayer(int fmt, const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd,
                     const float *x, int M, int H, int I,
                     double *y, double *g, double *u, double *h) {
    double *gg = (double *)malloc(sizeof(double) * (size_t)M * I);
    double *uu = (double *)malloc(sizeof(double) * (size_t)M * I);
    double *hh = (double *)malloc(sizeof(double) * (size_t)M * I);
    int8_t *xq = (int8_t *)malloc((size_t)M * H);
    float *xd = (float *)malloc(sizeof(float) * (size_t)M * (H / 32));
    int32_t *xs = (int32_t *)malloc(sizeof(int32_t) * (size_t)M * (H / 32));
    int8_t *hq = (int8_t *)malloc((size_t)M * I);
    float *hd = (float *)malloc(sizeof(float) * (size_t)M * (I / 32));
    int32_t *hs = (int32_t *)malloc(sizeof(int32_t) * (size_t)M * (I / 32));
    or_quantize_act(x, M, H, xq, xd, xs);
    or_gemv_q(fmt, Wg, xq, xd, xs, I, H, M, gg);
    or_gemv_q(fmt, Wu, xq, xd, xs, I, H, M, uu);
    for (size_t i = 0; i < (size_t)M * I; ++i) hh[i] = or_swiglu(gg[i], uu[i]);
    or_requant(hh, M, I, hq, hd, hs);
    or_gemv_q(fmt, Wd, hq, hd, hs, H, I, M, y);
    if (g) memcpy(g, gg, sizeof(double) * (size_t)M * I);
    if (u) memcpy(u, uu, sizeof(double) * (size_t)M * I);
    if (h) memcpy(h, hh, sizeof(double) * (size_t)M * I);
    free(gg); free(uu); free(hh); free(xq); free(xd); free(xs); free(hq); free(hd); free(hs);
}

/* ------------------------------------------------------------------------------------
 * Prefill GEMM on fp16 operands (readings in qg_oracle.h). */

/* From the definition of binary16: a finite nonzero value is r * 2^(e-10) with e the
 * exponent (clamped below at -14, where the spacing stops shrinking: gradual underflow)
 * and r an integer; r in [1024, 2048) is a normal number (exponent field e + 15,
 * fraction r - 1024), r < 1024 a subnormal one (exponent field 0, fraction r).  The
 * magnitude is scaled to units of 2^(e-10) exactly (a power-of-two scaling in fp64) and
 * rounded to the nearest integer, ties to the even one. */
uint16_t or_float_to_half(float f) {
    uint32_t bits;
    memcpy(&bits, &f, sizeof(bits));
    uint16_t sign = (uint16_t)((bits >> 31) << 15);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    if (isinf(f)) return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);          /* a = m * 2^E with m in [0.5, 1): a in [2^(E-1), 2^E) */
    int e = E - 1;
    if (e < -14) e = -14;
    double scaled = ldexp(a, 10 - e);
    double r = floor(scaled);
    double frac = scaled - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;
    if (r >= 2048.0) {     /* rounding carried into the next binade */
        r = 1024.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);  /* beyond 65504: infinity */
    if (r < 1024.0) return (uint16_t)(sign | (uint16_t)r);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(r - 1024.0));
}

void or_float_to_half_array(const float *x, size_t n, uint16_t *out) {
    for (size_t i = 0; i < n; ++i) out[i] = or_float_to_half(x[i]);
}

/* The fp16 weights of one row (K elements) by the reading: w32 = A*c - B*mc in fp32. */
static void dequant_row_f16(int fmt, const uint8_t *row, int K, uint16_t *out) {
    int QK = or_block_elems(fmt), BS = or_block_bytes(fmt);
    int32_t c[256], mc[256];
    double A[8], B[8];
    for (int b = 0; b < K / QK; ++b) {
        or_decode_block_mc(fmt, row + (size_t)b * BS, NULL, c, mc, A, B);
        for (int e = 0; e < QK; ++e) {
            float a32 = (float)A[e / 32], b32 = (float)B[e / 32];
            float p1 = a32 * (float)c[e];
            float p2 = b32 * (float)mc[e];
            float w32 = p1 - p2;
            out[(size_t)b * QK + e] = or_float_to_half(w32);
        }
    }
}

void or_dequant_f16(int fmt, const uint8_t *W, int N, int K, uint16_t *out) {
    size_t rb = (size_t)(K / or_block_elems(fmt)) * or_block_bytes(fmt);
    for (int n = 0; n < N; ++n) dequant_row_f16(fmt, W + (size_t)n * rb, K, out + (size_t)n * K);
}

void or_prefill_gemm(int fmt, const uint8_t *W, const float *x, int N, int K, int M, double *y, double *sabs) {
    size_t rb = (size_t)(K / or_block_elems(fmt)) * or_block_bytes(fmt);
    double *x16 = (double *)malloc(sizeof(double) * (size_t)M * K);
    for (size_t i = 0; i < (size_t)M * K; ++i) x16[i] = or_half_to_double(or_float_to_half(x[i]));
#pragma omp parallel for schedule(dynamic, 4) num_threads(or_get_threads())
    for (int n = 0; n < N; ++n) {
        uint16_t *w16 = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)K);
        double *wv = (double *)malloc(sizeof(double) * (size_t)K);
        dequant_row_f16(fmt, W + (size_t)n * rb, K, w16);
        for (int k = 0; k < K; ++k) wv[k] = or_half_to_double(w16[k]);
        for (int m = 0; m < M; ++m) {
            const double *xm = x16 + (size_t)m * K;
            double acc = 0.0, aabs = 0.0;
            for (int k = 0; k < K; ++k) {
                double p = wv[k] * xm[k];
                acc += p;
                aabs += fabs(p);
            }
            y[(size_t)m * N + n] = acc;
            if (sabs) sabs[(size_t)m * N + n] = aabs;
        }
        free(w16);
        free(wv);
    }
    free(x16);
}
