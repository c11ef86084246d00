/*
 * qg.h -- C ABI of libqg: decode-time GEMV computed in place on raw GGUF blocks,
 * with activations quantized on the GPU, plus the MoE FFN and the FFN sublayer
 * built from the same kernels.  Target: NVIDIA GB300 (sm_103a), one GPU.
 *
 * Sources (Chinese web pages, cited by title and section):
 *  [D27] "为什么专家缓存救不了稠密模型：16GB 显存跑 27B Dense 模型的推理优化实践"
 *        (xhh.club): section "原位量化计算与单流融合的实际收益" and the Q&A
 *        "如何让CUDA直接计算GGUF混合量化块而不展开为FP16？" -- GEMV directly on the
 *        GGUF blocks with no FP16 copy of W; activations quantized on the GPU to
 *        "Q8_F32S"; int8 dot products; K-quant correction term; I-quant codebook
 *        in registers; FFN sublayer on one stream with a reused workspace.
 *  [A3B] "参悟llama.cpp中的Qwen3.6-35B-A3B" (cnblogs), section 1.1: 256 experts,
 *        8 routed + 1 shared active per token, expert inter size 512, hidden 2048.
 *  [KES] "01 · 阶段总览：从 2B 到 8B 再到 MoE" (icman.com.cn): section 一 (a pure
 *        C ABI module whose device call returns 0 on success), section 二 issue ⑦
 *        (no cudaFree on the hot path: reuse buffers), section 四 issue ⑪ (router ->
 *        top-k -> expert gate/up -> swiglu -> down, weighted aggregation).
 *
 * Conventions for every call below:
 *  - All tensor pointers are owned by the caller.  Weights (W, the expert tensors, Wr)
 *    and the workspace ws must be device memory.  Activations and outputs (x, y, xq, xd,
 *    xs, topk_ids, topk_w, dots, aux) may be device memory or page-locked host memory
 *    that the device addresses directly (cudaHostAlloc / cudaHostRegister under unified
 *    addressing): the kernels then read and write them over the host link (NVLink-C2C on
 *    Grace systems) with no staging copy; results in host memory are complete when the
 *    stream reaches the point after the call.  The library never allocates, frees or
 *    synchronizes; each call only validates its arguments on the host and enqueues
 *    kernels on `stream` (a cudaStream_t; NULL = legacy default stream).
 *  - Return value: QG_OK (0) or a negative QG_E* status.  Every argument check happens
 *    on the host before any launch, so a failed call has enqueued nothing.  There is no
 *    CPU fallback: a GPU problem is reported, never silently computed elsewhere.
 *  - Layouts: x is M x K fp32 row-major; y is M x N fp32 row-major.  A weight matrix
 *    W with N rows and K columns is N rows of K/QK blocks each, rows contiguous, no
 *    padding, raw GGUF byte order.  QK = 32 elements for Q4_0, Q4_1, Q5_0, Q5_1, Q8_0
 *    and IQ4_NL; QK = 256 for Q2_K, Q3_K, Q4_K, Q5_K, Q6_K and IQ4_XS.  Expert tensors
 *    are E such matrices stacked contiguously.
 *  - Alignment: W and ws must be 16-byte aligned (QG_EALIGN otherwise); x, y and the
 *    quantized-activation arrays must be 4-byte aligned.
 *  - Limits: 1 <= M <= 16 tokens; K a positive multiple of the block size; N >= 1.
 *  - The workspace `ws` (device, caller-owned, >= qg_workspace_size(...) bytes) may be
 *    reused by back-to-back calls on the same stream; concurrent calls on different
 *    streams need separate workspaces.
 */
#ifndef QG_H
#define QG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Block formats, numbered by their GGUF type ids. */
enum qg_format {
    QG_Q4_0 = 2,    /* 32 elements, 18 B: fp16 d, 16 B of 4-bit codes; w = d*(c-8)           */
    QG_Q4_1 = 3,    /* 32 elements, 20 B: fp16 d, fp16 m, 4-bit codes; w = d*c + m           */
    QG_Q5_0 = 6,    /* 32 elements, 22 B: fp16 d, 32 fifth bits, 4-bit codes; w = d*(c-16)   */
    QG_Q5_1 = 7,    /* 32 elements, 24 B: fp16 d, fp16 m, fifth bits, codes; w = d*c + m     */
    QG_Q8_0 = 8,    /* 32 elements, 34 B: fp16 d, 32 int8 codes; w = d*q                     */
    QG_Q2_K = 10,   /* 256 elements, 84 B: 16 x (4-bit scale, 4-bit min), 2-bit codes, d, dmin */
    QG_Q3_K = 11,   /* 256 elements, 110 B: 3-bit codes (2 low + 1 high), 16 6-bit scales, d */
    QG_Q4_K = 12,   /* 256 elements, 144 B: fp16 d, dmin, 8 x 6-bit scale/min, 4-bit codes   */
    QG_Q5_K = 13,   /* 256 elements, 176 B: as Q4_K plus one high bit per code              */
    QG_Q6_K = 14,   /* 256 elements, 210 B: 6-bit codes, 16 int8 sub-scales, fp16 d          */
    QG_IQ4_NL = 20, /* 32 elements, 18 B: fp16 d, 4-bit indices into the 16-entry codebook   */
    QG_IQ4_XS = 23  /* 256 elements, 136 B: fp16 d, 6-bit sub-scales, 4-bit codebook indices */
};

/* Status codes. */
enum qg_status {
    QG_OK = 0,
    QG_EINVAL = -1,     /* bad format, shape, token count, pointer or top-k           */
    QG_EWORKSPACE = -2, /* ws is NULL or ws_bytes is below qg_workspace_size()         */
    QG_EALIGN = -3,     /* a pointer breaks the alignment rule above                   */
    QG_ECUDA = -4,      /* a CUDA runtime call or kernel launch failed                 */
    QG_EDEVICE = -5     /* the current device is not an sm_103 GPU the library targets */
};

/* Operations for qg_workspace_size(). */
enum qg_op {
    QG_OP_GEMV = 1,
    QG_OP_GEMV_Q = 2,
    QG_OP_MOE_FFN = 3,
    QG_OP_FFN_SUBLAYER = 4,
    QG_OP_MOE_FFN_S16 = 5,
    QG_OP_PREFILL = 6
};

/* Activation quantization "Q8_F32S" [D27 Q&A]: for each token m and each 32-element
 * block b of K, d = amax|x| / 127 (fp32, IEEE division), q = clamp(roundf(x / d),
 * -127, 127) with round-half-away-from-zero (all q = 0 and d = 0 for an all-zero
 * block), s = sum of the 32 codes.
 *   x:  M x K fp32.   xq: M x K int8.   xd: M x K/32 fp32.   xs: M x K/32 int32.
 * K must be a multiple of 32. */
int qg_quantize_act(const float *x, int M, int K, int8_t *xq, float *xd, int32_t *xs, void *stream);

/* s16 activation quantization [KES section 四, issue ⑫: int8 activation error compounds
 * over many MoE layers; the MoE FFN moved to s16 activations with a step 256 times finer]:
 * the rule of qg_quantize_act with d = amax|x| / 32512 (= (amax / 127) / 256, fp32 IEEE
 * division) and q = clamp(roundf(x / d), -32512, 32512).
 *   x: M x K fp32.   xq: M x K int16 (2-byte aligned).   xd: M x K/32 fp32.
 *   xs: M x K/32 int32 (sum of the 32 codes).  K must be a multiple of 32.
 * The MoE's s16 path (qg_moe_ffn_s16) computes the same codes on the fly; this call is
 * the plain-layout form, for callers and tests. */
int qg_quantize_act_s16(const float *x, int M, int K, int16_t *xq, float *xd, int32_t *xs, void *stream);

/* y = W x for M tokens [D27 Q&A; KES section 一]: x is quantized on the GPU as by
 * qg_quantize_act (once per call, into per-task activation tiles in ws), then each
 * 32-element unit u (activation step xd, code sum xs) contributes
 *   Q8_0, Q4_0, Q5_0, IQ4_NL:  y += d * xd * dot
 *   Q6_K, Q3_K:                y += d * xd * dot   (the 16-element sub-scales are in dot)
 *   IQ4_XS:                    y += d*(ls_u - 32) * xd * dot
 *   Q4_1, Q5_1:                y += xd * (d * dot + m * xs)
 *   Q4_K, Q5_K:                y += xd * (d*S_j * dot - dmin*M_j * xs)
 *   Q2_K:                      y += xd * (d * dot - dmin * mins)
 * where dot is the exact int32 sum of weight codes times activation codes, with the
 * codes of qg_block_dots below (its offsets included: nibble-8, code-16, code-32, the
 * codebook value), and mins is the exact sum of each 16-element sub-block's 4-bit min
 * times its activation codes.
 *   fmt: qg_format.  W: N x K blocks.  x: M x K fp32.  y: M x N fp32 (overwritten). */
int qg_gemv(int fmt, const void *W_blocks, const float *x, float *y, int N, int K, int M,
            void *ws, size_t ws_bytes, void *stream);

/* Same as qg_gemv with the activations already quantized (xq, xd, xs laid out as
 * produced by qg_quantize_act).  Both GEMV calls need a workspace (ws != NULL). */
int qg_gemv_q(int fmt, const void *W_blocks, const int8_t *xq, const float *xd, const int32_t *xs,
              float *y, int N, int K, int M, void *ws, size_t ws_bytes, void *stream);

/* Bytes of the library's fixed device scratch array used by qg_gemv_static_ws. */
#define QG_STATIC_WS_BYTES 2097152

/* qg_gemv without a caller workspace.  The pages have no counterpart to this entry point.
 * It is for callers that cannot allocate device memory at the point where they call the
 * GEMV: code running inside a host framework whose allocator owns all device memory (a
 * plugin must not call cudaMalloc behind its back), code on a latency-critical path where
 * cudaMalloc's implicit device synchronization is not acceptable, or a plain C host
 * program that links only this library and has no device allocator of its own.  Such a
 * caller passes only its inputs and outputs; the scratch lives in one file-scope device
 * array of QG_STATIC_WS_BYTES bytes inside the library, held by every GPU that loads the
 * library until the process exits.  The call itself allocates nothing.
 *   Arguments, layouts and results as qg_gemv (y is bit-identical to qg_gemv's).
 *   Limit: returns QG_EWORKSPACE, without launching, when qg_workspace_size(QG_OP_GEMV,
 *   fmt, M, N, K, ...) exceeds QG_STATIC_WS_BYTES (e.g. very long rows at M = 16).
 *   Contents: the array keeps whatever the last call left in it; every call writes all
 *   of the scratch it reads before reading it, so nothing needs to start at zero.
 *   Races: every call on a device shares the one array.  Calls whose executions may
 *   overlap on the GPU (different streams without ordering, or several host threads)
 *   corrupt each other's activations; order them on one stream.
 *   Set-up: the first call in each CUDA context of a device looks up the array's device
 *   address (cudaGetSymbolAddress, with that device current); make that first call before
 *   any stream capture.  The address is cached per device together with the context's id
 *   and looked up again when the device's context has changed (after cudaDeviceReset, or
 *   when a host framework re-creates the primary context). */
int qg_gemv_static_ws(int fmt, const void *W_blocks, const float *x, float *y, int N, int K, int M,
                      void *stream);

/* MoE FFN for M tokens [KES section 四 ⑪; A3B section 1.1]:
 *   logits = Wr x (fp32); probabilities = softmax over the E experts; the topk largest
 *   (ties: lower expert id) are renormalized to weights w summing to 1;
 *   for each routed slot and for the shared expert: g = Wg x, u = Wu x (x quantized
 *   once per token), h = silu(g) * u, h requantized per 32 as in qg_quantize_act,
 *   o = Wd h; y = sum over routed slots (in rank order) of w * o, plus 1.0 * o of the
 *   shared expert (ungated).
 *   x: M x H fp32.  Wr: E x H fp32.  Wg_exps, Wu_exps: E stacked I x H matrices;
 *   Wd_exps: E stacked H x I matrices.  Wg_sh, Wu_sh: I x H; Wd_sh: H x I.
 *   y: M x H fp32.  topk_ids (int32) / topk_w (fp32): M x topk, may be NULL.
 *   Limits: 1 <= topk <= 16, topk <= E <= 1024, H and I multiples of the block size, and
 *   the activation tiles of all M tokens over H within one CTA's 140 KB tile area (about
 *   1.5 bytes per element and token: every M up to 16 for H <= 4096; M <= 13 for H = 7168
 *   with Q4_K); QG_EINVAL otherwise, before any launch (qg_workspace_size returns
 *   (size_t)-1 for such a shape).
 * The intermediates stay in ws; qg_moe_ws_layout() gives their offsets. */
int qg_moe_ffn(int fmt, const float *x, int M, int H,
               const float *Wr, int E, int topk,
               const void *Wg_exps, const void *Wu_exps, const void *Wd_exps,
               const void *Wg_sh, const void *Wu_sh, const void *Wd_sh, int I,
               float *y, int32_t *topk_ids, float *topk_w,
               void *ws, size_t ws_bytes, void *stream);

/* The MoE FFN with s16 activations [KES section 四, issue ⑫]: as qg_moe_ffn, with x and
 * the requantized h quantized by the qg_quantize_act_s16 rule instead of the int8 one (the
 * router still reads fp32 x).  Arguments, layouts, limits and errors as qg_moe_ffn (the
 * tile-area limit counts two planes per token: every M up to 16 for H <= 2048); the
 * workspace is qg_workspace_size(QG_OP_MOE_FFN_S16, ...) and its intermediates are at
 * qg_moe_s16_ws_layout().  On the GPU an s16 code q is held as two int8 planes,
 * q = 256 * hi + lo, whose exact integer dots are combined in fp32: twice the dot work
 * and activation traffic of the int8 path over the same weight bytes. */
int qg_moe_ffn_s16(int fmt, const float *x, int M, int H,
                   const float *Wr, int E, int topk,
                   const void *Wg_exps, const void *Wu_exps, const void *Wd_exps,
                   const void *Wg_sh, const void *Wu_sh, const void *Wd_sh, int I,
                   float *y, int32_t *topk_ids, float *topk_w,
                   void *ws, size_t ws_bytes, void *stream);

/* FFN sublayer on one stream with a reused workspace [D27 section
 * "原位量化计算与单流融合的实际收益"]: x quantized once, g = Wg x and u = Wu x in one
 * launch, h = silu(g) * u, h requantized, y = Wd h.
 *   Wg, Wu: I x H blocks; Wd: H x I blocks; x: M x H fp32; y: M x H fp32. */
int qg_ffn_sublayer(int fmt, const void *Wg, const void *Wu, const void *Wd,
                    const float *x, float *y, int M, int H, int I,
                    void *ws, size_t ws_bytes, void *stream);

/* Prefill GEMM on the tensor cores over raw blocks [KES section 九: prefill moved to the
 * tensor cores with the weights dequantized to fp16 inside the kernel; section 四, issue ⑮:
 * prefill takes float activations, not int8 ones], for M tokens at once (M >> 16):
 *   y[m][n] = sum_k fp16(w[n][k]) * fp16(x[m][k]), accumulated in fp32, where
 *   w[n][k] is formed per 32-element unit in fp32 as A_u * c_e - B_u * mc_e (the factors and
 *   codes of qg_block_dots: both products exact, one rounding) and rounded to the nearest
 *   fp16 (ties to even), and fp16(x) is the nearest fp16 of x (ties to even).
 *   fmt: qg_format.  W: N x K blocks (16-byte aligned).  x: M x K fp32.  y: M x N fp32.
 *   Limits: 1 <= M <= 1048576 (QG_EINVAL otherwise); K a multiple of the block size.
 *   ws: device, >= qg_workspace_size(QG_OP_PREFILL, fmt, M, N, K, 0, 0, 0) bytes, 16-byte
 *   aligned: the fp16 activation tiles (about 2 x M x K bytes) and, for K-split shapes,
 *   fp32 partial sums.  |x| beyond 65504 rounds to infinity in fp16 (the caller's range).
 * Launches a conversion kernel, the tensor-core kernel (tcgen05.mma, fp32 accumulators in
 * tensor memory) and, for K-split shapes, a reduction; asynchronous on stream like every
 * call here. */
int qg_prefill_gemm(int fmt, const void *W_blocks, const float *x, float *y, int N, int K, int M,
                    void *ws, size_t ws_bytes, void *stream);

/* Test hook of the prefill operand: out[n][k] = the fp16 bit pattern of w[n][k] as formed by
 * qg_prefill_gemm (same device decoders).  out: N x K uint16, device memory (or page-locked
 * host memory), 4-byte aligned. */
int qg_dequant_f16(int fmt, const void *W_blocks, int N, int K, uint16_t *out, void *stream);

/* Bytes of workspace an operation needs; 0 means the call needs none (ws may then be
 * NULL); (size_t)-1 means the arguments are invalid.  The size depends on the shape and
 * on the current device's SM count (152 is assumed when no device is usable).
 *   QG_OP_GEMV / QG_OP_GEMV_Q: (fmt, M, N, K)            E, topk, I ignored
 *   QG_OP_MOE_FFN, QG_OP_MOE_FFN_S16: (fmt, M, N=H, K=H, E, topk, I)
 *   QG_OP_FFN_SUBLAYER:        (fmt, M, N=H, K=H, I)      E, topk ignored
 *   QG_OP_PREFILL:             (fmt, M, N, K)             E, topk, I ignored */
size_t qg_workspace_size(int op, int fmt, int M, int N, int K, int E, int topk, int I);

/* Offsets (bytes from ws) of the MoE intermediates, written by qg_moe_ffn:
 *   off[0] g, off[1] u, off[2] h : fp32, M x (topk+1) x I (slot topk = shared expert)
 *   off[3] hq (int8), off[4] hd (fp32), off[5] hs (int32): requantized h,
 *          M x (topk+1) x I  and  M x (topk+1) x I/32
 *   off[6] logits: fp32 M x E
 * Returns QG_OK or QG_EINVAL. */
int qg_moe_ws_layout(int M, int H, int E, int topk, int I, size_t off[7]);

/* The same offsets for qg_moe_ffn_s16, whose intermediates are:
 *   off[0] g, off[1] u : fp32, M x (topk+1) x 2 x I -- per row the two planes' partial
 *          results, whose fp32 sum is g (u)
 *   off[2] h : fp32, M x (topk+1) x I
 *   off[3] hq (int16), off[4] hd (fp32), off[5] hs (int32): h requantized by the s16 rule,
 *          M x (topk+1) x I  and  M x (topk+1) x I/32
 *   off[6] logits: fp32 M x E */
int qg_moe_s16_ws_layout(int M, int H, int E, int topk, int I, size_t off[7]);

/* Offsets of the FFN sublayer intermediates: off[0] g, off[1] u, off[2] h (fp32 M x I). */
int qg_ffn_ws_layout(int fmt, int M, int H, int I, size_t off[3]);

/* Test hook, exact integer contract: dots[m][n][u] = sum over the 32 elements of unit
 * u of (weight code) * xq, where the weight code is q (Q8_0), nibble-8 (Q4_0), the
 * unsigned code (Q4_1, Q5_1, Q4_K, Q5_K), 5-bit code-16 (Q5_0), sub-scale*code (Q2_K),
 * (scale-32)*(signed 3-bit code) (Q3_K), sub-scale*(code-32) (Q6_K) or the codebook
 * value (IQ4_NL, IQ4_XS); aux[m][n][u] = the unit's min sum for the formats with a min
 * term: xs[m][u] for Q4_1, Q5_1, Q4_K, Q5_K, and sum of (16-element sub-block min) * xq
 * for Q2_K; else 0.  dots, aux: M x N x K/32 int32.  Uses the same block decoders as the
 * GEMV kernels. */
int qg_block_dots(int fmt, const void *W_blocks, const int8_t *xq, const int32_t *xs,
                  int N, int K, int M, int32_t *dots, int32_t *aux, void *stream);

/* Device-side error word, read and cleared: value 1 = a bounded wait in a kernel gave up
 * (results of that call are invalid); value 2 = a launch plan did not fit the engine's
 * per-stage piece table and some rows were skipped (a library bug; results invalid).
 * Synchronizes the current device; for tests and diagnostics, not for the hot path. */
int qg_device_error(unsigned int *err);

/* Test hook of the failure detector (bounded waits): launches one thread that waits,
 * through the same bounded wait routine as every kernel here, for an mbarrier phase that
 * never completes, with a limit of limit_ns (1 us to 1 s; QG_EINVAL otherwise).  The wait
 * gives up, records value 1 in the device error word (qg_device_error) and the kernel
 * returns: the context stays usable.  Asynchronous on stream. */
int qg_test_wait_expiry(unsigned long long limit_ns, void *stream);

/* Human-readable text of a status code. */
const char *qg_strerror(int status);

/* Library version (major*10000 + minor*100 + patch). */
int qg_version(void);

#ifdef __cplusplus
}
#endif
#endif /* QG_H */
