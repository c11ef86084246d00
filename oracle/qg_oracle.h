/*
 * qg_oracle.h -- plain, slow CPU oracle for the quantized decode GEMV over raw
 * GGUF blocks, the MoE FFN built on it and the FFN sublayer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no source with the CUDA library.
 *
 * Sources (page titles as printed; the pages are Chinese web pages):
 *  [D27]  "为什么专家缓存救不了稠密模型：16GB 显存跑 27B Dense 模型的推理优化实践"
 *         (xhh.club) -- "延伸解读 / 原位量化计算与单流融合的实际收益" and the
 *         Q&A "如何让CUDA直接计算GGUF混合量化块而不展开为FP16？": GEMV on the raw
 *         GGUF blocks, activations quantized to "Q8_F32S", int8 dot products,
 *         K-quant correction term, I-quant codebook in registers.
 *  [A3B]  "参悟llama.cpp中的Qwen3.6-35B-A3B" (cnblogs) -- section 1.1: 256
 *         experts, 8 routed + 1 shared active, expert inter size 512, hidden 2048.
 *  [KES]  "01 · 阶段总览：从 2B 到 8B 再到 MoE" (icman.com.cn) -- section 四,
 *         issue ⑪: router -> top-k -> expert gate/up -> swiglu -> down, weighted
 *         aggregation; section 九 "CPU 对照": a CPU reference that dequantizes
 *         q8/q4 rows and takes dot products.
 *
 * The pages name the block formats but never print their byte layouts; the
 * layouts used here are the public GGUF block definitions.  Readings taken where
 * the pages are silent are stated next to the code that takes them.
 *
 * Parity unpinned: the 16 values of the IQ4_NL codebook used by IQ4_XS.  The pages
 * print no table (they only say the codebook is small and lives in registers); the
 * values are the published IQ4_NL table, and a test can only restate them.  The
 * decode of IQ4_XS around the table (indices, sub-scales, d) is pinned.  Agreement of
 * the twelve byte layouts with real GGUF files is likewise unpinned: no file is at hand.
 *
 * All floating point here is fp64 unless the method itself fixes fp32 (the
 * activation scale and the division that produces the activation codes).
 */
#ifndef QG_ORACLE_H
#define QG_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GGUF type ids of the block formats. */
enum {
    OR_Q4_0 = 2, OR_Q4_1 = 3, OR_Q5_0 = 6, OR_Q5_1 = 7, OR_Q8_0 = 8,
    OR_Q2_K = 10, OR_Q3_K = 11, OR_Q4_K = 12, OR_Q5_K = 13, OR_Q6_K = 14, OR_IQ4_NL = 20, OR_IQ4_XS = 23
};

/* Elements per block (32 or 256) and bytes per block; 0 for an unknown format. */
int or_block_elems(int fmt);
int or_block_bytes(int fmt);

/* IEEE binary16 (little-endian bit pattern) to double, exact. */
double or_half_to_double(uint16_t h);

/* Decode one block.  w[QK]: the dequantized weights (fp64).  c[QK]: the integer
 * codes of the per-32 dot-product contract (Q8_0: q; Q4_0: nibble-8; Q4_1: nibble;
 * Q5_0: 5-bit code - 16; Q5_1: 5-bit code; Q4_K/Q5_K: unsigned code;
 * Q6_K: sc[e/16]*(code-32); Q2_K: sc[e/16]*code; Q3_K: (scale-32)*(code-4 or code);
 * IQ4_XS, IQ4_NL: codebook value).  mc[QK]: the integer min codes (Q2_K: the 4-bit
 * min of the element's 16-element sub-block; 1 for every other format).
 * A[QK/32], B[QK/32]: per 32-element unit, the factors with
 *   w_e = A_u * c_e - B_u * mc_e  (Q6_K, Q3_K: B_u = 0, the sub-scale is in c_e)
 * Any output pointer may be NULL. */
void or_decode_block(int fmt, const uint8_t *blk, double *w, int32_t *c, double *A, double *B);
void or_decode_block_mc(int fmt, const uint8_t *blk, double *w, int32_t *c, int32_t *mc, double *A, double *B);

/* Dequantize a whole N x K matrix to fp64 (row-major). */
void or_dequant_matrix(int fmt, const uint8_t *W, int N, int K, double *out);

/* Activation quantization ("Q8_F32S"): per token, per 32 consecutive elements,
 * d = amax/127 (fp32 division), q = clamp(roundf(x/d), -127, 127), s = sum q.
 * x: M x K fp32.  xq: M x K int8.  xd, xs: M x K/32.  K must be a multiple of 32. */
void or_quantize_act(const float *x, int M, int K, int8_t *xq, float *xd, int32_t *xs);

/* s16 activations ([KES] section 四, issue ⑫): the same rule with a step 256 times finer,
 * d = amax/32512 (fp32 division; equal to (amax/127)/256), q = clamp(roundf(x/d),
 * -32512, 32512), s = sum q.  xq: M x K int16. */
void or_quantize_act16(const float *x, int M, int K, int16_t *xq, float *xd, int32_t *xs);

/* Per-32 integer dot products: dots[m][n][u] = sum_i c_i * xq[m][32u+i];
 * aux[m][n][u] = sum_i mc_i * xq[m][32u+i] (= xs[m][u] where mc = 1) for the formats
 * with a min term (Q4_1, Q5_1, Q2_K, Q4_K, Q5_K), else 0.  Layout M x N x (K/32). */
void or_block_dots(int fmt, const uint8_t *W, const int8_t *xq, const int32_t *xs,
                   int N, int K, int M, int32_t *dots, int32_t *aux);

/* y[m][n] = sum_u xd[m][u] * (A_u * dot - B_u * aux) in fp64 from the integer sums,
 * aux = xs[m][u] (Q2_K: the sum over the unit of mc_i * xq, with its per-16 mins)
 * (the exact result the GPU path reaches up to rounding order). */
void or_gemv_q(int fmt, const uint8_t *W, const int8_t *xq, const float *xd, const int32_t *xs,
               int N, int K, int M, double *y);
/* The same with s16 activation codes. */
void or_gemv_q16(int fmt, const uint8_t *W, const int16_t *xq, const float *xd, const int32_t *xs,
                 int N, int K, int M, double *y);

/* Same y by brute force: fp64 dequantize-then-dot against xhat = q*d. */
void or_gemv_deq(int fmt, const uint8_t *W, const int8_t *xq, const float *xd,
                 int N, int K, int M, double *y);

/* sabs[m][n] = sum_k |w_k * xhat_k|, the scale of the per-element tolerance. */
void or_absdot(int fmt, const uint8_t *W, const int8_t *xq, const float *xd,
               int N, int K, int M, double *sabs);
void or_absdot16(int fmt, const uint8_t *W, const int16_t *xq, const float *xd,
                 int N, int K, int M, double *sabs);

/* Full GEMV: quantize x, then or_gemv_q.  y: M x N. */
void or_gemv(int fmt, const uint8_t *W, const float *x, int N, int K, int M, double *y);

/* Router: logits = Wr x (fp64 from fp32 inputs), softmax over E (max-subtracted),
 * top-k by probability (ties: lower expert id first), weights renormalized over
 * the k picks.  x: M x H; Wr: E x H row-major.  Outputs may be NULL except ids/w:
 * logits, probs: M x E; ids: M x topk; w: M x topk (fp64). */
void or_router(const float *x, int M, int H, const float *Wr, int E, int topk,
               double *logits, double *probs, int32_t *ids, double *w);

/* silu(g) * u = g * u / (1 + exp(-g)). */
double or_swiglu(double g, double u);

/* MoE gate/up stage for the slots of each token: slot s < topk uses routed expert
 * ids[m][s]; slot topk is the shared expert.  Expert tensors are E matrices stacked
 * contiguously (gate/up: I x H each; down: H x I each).  x is quantized once per token.
 * g, u, h: M x (topk+1) x I (fp64).  x_q/xd/xs may be NULL (then quantized here). */
void or_moe_gateup(int fmt, const float *x, int M, int H, int E, int topk, int I,
                   const int32_t *ids, const uint8_t *Wg_exps, const uint8_t *Wu_exps,
                   const uint8_t *Wg_sh, const uint8_t *Wu_sh,
                   double *g, double *u, double *h);

/* Requantize h: round each fp64 h to fp32, then the activation quantization rule.
 * h: R x I; hq: R x I; hd, hs: R x I/32. */
void or_requant(const double *h, int R, int I, int8_t *hq, float *hd, int32_t *hs);

/* MoE down stage: o[m][s] = Wd_{slot expert} . hq[m][s]; y[m] = sum_{s<topk} w[m][s]*o[m][s]
 * + 1.0 * o[m][topk] (shared, ungated), summed in slot order.  hq: M x (topk+1) x I.
 * y: M x H.  o (nullable): M x (topk+1) x H.  yabs (nullable): the same sum over
 * |w| * sum|w_k * hhat_k|, for the tolerance. */
void or_moe_down(int fmt, int M, int H, int E, int topk, int I,
                 const int32_t *ids, const double *w,
                 const int8_t *hq, const float *hd, const int32_t *hs,
                 const uint8_t *Wd_exps, const uint8_t *Wd_sh,
                 double *y, double *o, double *yabs);

/* Whole MoE FFN: route, gate/up, swiglu, requant, down, weighted sum.  ids/w are
 * outputs (M x topk). */
void or_moe_ffn(int fmt, const float *x, int M, int H, const float *Wr, int E, int topk,
                const uint8_t *Wg_exps, const uint8_t *Wu_exps, const uint8_t *Wd_exps,
                const uint8_t *Wg_sh, const uint8_t *Wu_sh, const uint8_t *Wd_sh, int I,
                double *y, int32_t *ids, double *w);

/* The MoE FFN and its stages with s16 activations ([KES] section 四, issue ⑫): x and
 * the requantized h both follow or_quantize_act16; the router is unchanged (fp32 x). */
void or_moe_gateup16(int fmt, const float *x, int M, int H, int E, int topk, int I,
                     const int32_t *ids, const uint8_t *Wg_exps, const uint8_t *Wu_exps,
                     const uint8_t *Wg_sh, const uint8_t *Wu_sh,
                     double *g, double *u, double *h);
void or_requant16(const double *h, int R, int I, int16_t *hq, float *hd, int32_t *hs);
void or_moe_down16(int fmt, int M, int H, int E, int topk, int I,
                   const int32_t *ids, const double *w,
                   const int16_t *hq, const float *hd, const int32_t *hs,
                   const uint8_t *Wd_exps, const uint8_t *Wd_sh,
                   double *y, double *o, double *yabs);
void or_moe_ffn16(int fmt, const float *x, int M, int H, const float *Wr, int E, int topk,
                  const uint8_t *Wg_exps, const uint8_t *Wu_exps, const uint8_t *Wd_exps,
                  const uint8_t *Wg_sh, const uint8_t *Wu_sh, const uint8_t *Wd_sh, int I,
                  double *y, int32_t *ids, double *w);

/* FFN sublayer: quantize x, g = Wg x, u = Wu x (Wg, Wu: I x H), h = silu(g)*u,
 * requantize h, y = Wd h (Wd: H x I).  g, u, h (nullable): M x I. */
void or_ffn_sublayer(int fmt, const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd,
                     const float *x, int M, int H, int I,
                     double *y, double *g, double *u, double *h);

/* ---------------------------------------------------------------------------------
 * Prefill GEMM on fp16 operands ([KES] section 九: the prefill matrix products moved to
 * the tensor cores with the weights dequantized to fp16 inside the kernel, prefill of 512
 * tokens 372 -> 902 tokens/s; section 四, issue ⑮: prefill takes float activations, not
 * int8 ones, because int8 activations cost ten times the perplexity there).  Readings:
 *  - each weight is formed in fp32 from its block, w32 = A_u * c_e - B_u * mc_e with the
 *    factors of or_decode_block_mc (both products are exact in fp32 for every format
 *    here; the subtraction rounds once), then rounded to the nearest fp16, ties to even;
 *  - each activation is its fp32 value rounded to the nearest fp16, ties to even;
 *  - y[m][n] = sum_k w16[n][k] * x16[m][k]; the oracle sums the exact products in fp64
 *    (the GPU accumulates in fp32).
 * Parity of these readings against the page's own kernel is unpinned: the page prints
 * neither its rounding nor its dequantization order. */

/* IEEE binary32 -> binary16, round to nearest, ties to even (overflow to infinity,
 * gradual underflow, NaN kept as a quiet NaN).  Returns the binary16 bit pattern. */
uint16_t or_float_to_half(float f);
void or_float_to_half_array(const float *x, size_t n, uint16_t *out);

/* fp16 weights of an N x K matrix (bit patterns, row-major), by the reading above. */
void or_dequant_f16(int fmt, const uint8_t *W, int N, int K, uint16_t *out);

/* y[m][n] = sum_k w16[n][k] * x16[m][k] in fp64 (x: M x K fp32; y: M x N).
 * sabs (nullable): sum_k |w16 * x16|, the scale of the per-element tolerance. */
void or_prefill_gemm(int fmt, const uint8_t *W, const float *x, int N, int K, int M, double *y, double *sabs);

/* Threads used by the OpenMP loops over output rows (1 = single-threaded). */
void or_set_threads(int n);
int or_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
