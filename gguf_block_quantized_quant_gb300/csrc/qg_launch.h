// qg_launch.h -- host interface between the C ABI (qg_abi.cu) and the per-format
// launchers (qg_fmt.cu, compiled once per block format).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "qg_plan.h"

namespace qg {

struct GemvCall {
    const uint8_t *W;
    int N, K, M;
    const float *x;     // fp32 activations, or NULL when xq/xd/xs are given
    const float *u;     // optional: the activations are silu(x) * u (written to h_out if set)
    float *h_out;
    const int8_t *xq;
    const float *xd;
    const int32_t *xs;
    float *y;
    uint8_t *ws;
    size_t ws_bytes;
    cudaStream_t stream;
    bool x_device;      // x is device memory (not host memory mapped for the device)
};

struct FfnCall {
    const uint8_t *Wg, *Wu, *Wd;
    const float *x;
    float *y;
    int M, H, I;
    uint8_t *ws;
    size_t ws_bytes;
    cudaStream_t stream;
    bool x_device;  // x is device memory
};

struct MoeCall {
    const float *x;
    int M, H;
    const float *Wr;
    int E, topk;
    const uint8_t *Wg_exps, *Wu_exps, *Wd_exps, *Wg_sh, *Wu_sh, *Wd_sh;
    int I;
    float *y;
    int32_t *ids_out;
    float *w_out;
    bool s16;           // s16 activations (two int8 planes per activation row)
    uint8_t *ws;
    size_t ws_bytes;
    cudaStream_t stream;
};

struct DotsCall {
    const uint8_t *W;
    const int8_t *xq;
    const int32_t *xs;
    int N, K, M;
    int32_t *dots, *aux;
    cudaStream_t stream;
};

struct PrefillCall {
    const uint8_t *W;
    const float *x;     // M x K fp32
    float *y;           // M x N fp32
    int N, K, M;
    uint8_t *ws;
    size_t ws_bytes;
    cudaStream_t stream;
};

// Per-format launchers (status codes as in qg.h).
template <int FMT>
int gemv_run(const GemvCall &c, int sms);
template <int FMT>
int gemv_run_planned(const GemvPlan &p, const GemvCall &c);
template <int FMT>
int ffn_run(const FfnCall &c, int sms);
template <int FMT>
int moe_run(const MoeCall &c, int sms);
template <int FMT>
int dots_run(const DotsCall &c);
template <int FMT>
int dev_err_take(unsigned int *err);  // read and clear the format's device error word
template <int FMT>
int prefill_run(const PrefillCall &c, int sms);
template <int FMT>
int dequant_f16_run(const uint8_t *W, int N, int K, uint16_t *out, cudaStream_t s);

// Format-independent kernels (qg_abi.cu).
int launch_quant_act(const float *x, int M, int K, long ldx, int8_t *xq, float *xd, int32_t *xs,
                     cudaStream_t s);
int launch_splitk_reduce(const float *part, int KS, long MN, float *y, cudaStream_t s);
// Activation tile image of `rows` rows of K elements (tiles of 2^xgt_log2 activation blocks),
// from fp32 rows x (quantized here; with u != NULL the rows are silu(x) * u, also written to
// h_out when given) or from xq/xd/xs; mq/md/ms optionally receive the quantized rows in
// their plain layout.
int launch_prep_tiles(const float *x, const float *u, float *h_out, const int8_t *xq, const float *xd,
                      const int32_t *xs, int rows, int K, int xgt_log2, uint8_t *img, int8_t *mq, float *md,
                      int32_t *ms, cudaStream_t s);
// fp16 activation image of the prefill GEMM: M x K fp32 rows -> nkt tiles of 64 elements x
// ntt tiles of BT tokens (K tile major), each BT x 128 bytes in the tensor cores' K-major
// 128-byte-swizzled layout (rows past M and elements past K are zero).
int launch_prefill_x16(const float *x, int M, int K, int BT, int ntt, int nkt, uint8_t *img, cudaStream_t s);
// Router logits (fp32) and the activation tile image of x (s16: two planes per row) in one
// launch.
int launch_router_prep(const float *x, int M, int H, const float *Wr, int E, float *logits, int xgt_log2,
                       uint8_t *img, bool s16, cudaStream_t s);

}  // namespace qg
