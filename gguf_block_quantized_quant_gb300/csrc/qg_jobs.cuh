// qg_jobs.cuh -- stage sequences, activation sources, prologues and epilogues of the
// four GEMV-shaped operations run by the streaming engine (qg_engine.cuh):
//
//   GemvJob       y = W x (optionally one K-slice per CTA, partial sums to a buffer)
//   FfnGateUpJob  g = Wg x, u = Wu x in one pass over both matrices, h = silu(g)*u
//   MoeGateUpJob  the same for each token's routed experts and the shared expert, with
//                 the softmax/top-k of the router computed by the producer warp
//   MoeDownJob    o = Wd_e h for every slot, y = sum_routed w*o + o_shared (slot order)
#pragma once

#include <type_traits>

#include "qg_engine.cuh"

namespace qg {

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Consumers quantize `rows` activation rows of `cols` fp32 values (cols a multiple of 32)
// into shared memory: codes at q + r*ldq + c, scales/sums at d/s + 4*(r*lds + c/32).
// Optionally mirror the result to global memory (gq/gd/gs, row pitch cols).
__device__ __forceinline__ void quantize_rows_to_smem(const float *src, long src_ld, int rows, int cols,
                                                      uint32_t q, uint32_t d, uint32_t s, int ldq, int lds,
                                                      int tid, int8_t *gq, float *gd, int32_t *gs) {
    const int warp = tid >> 5, lane = tid & 31;
    const int nb = cols / 32;
    for (int w = warp; w < rows * nb; w += NCW) {
        const int r = w / nb, b = w - r * nb;
        const float v = src[(long)r * src_ld + 32 * b + lane];
        int qi, si;
        float di;
        quant_block_warp(v, qi, di, si);
        sts8(q + (uint32_t)(r * ldq + 32 * b + lane), (uint32_t)qi & 255u);
        if (gq) gq[(long)r * cols + 32 * b + lane] = (int8_t)qi;
        if (lane == 0) {
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(d + 4u * (uint32_t)(r * lds + b)), "f"(di) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(s + 4u * (uint32_t)(r * lds + b)), "r"(si) : "memory");
            if (gd) {
                gd[(long)r * nb + b] = di;
                gs[(long)r * nb + b] = si;
            }
        }
    }
}

// Byte offsets of a quantized-activation area inside a job's shared memory.
struct XArea {
    uint32_t q, d, s, bytes;
    int ldq, lds;
};
__host__ __device__ inline XArea make_xarea(uint32_t base, int rows, int cols) {
    XArea a;
    a.ldq = cols;
    a.lds = cols / 32;
    a.q = base;
    a.d = base + (uint32_t)(((long)rows * cols + 15) / 16 * 16);
    a.s = a.d + 4u * (uint32_t)(rows * a.lds);
    a.bytes = a.s + 4u * (uint32_t)(rows * a.lds) - base;
    return a;
}

// ===================================================================================== GEMV
template <int FMT, bool XSM>
struct GemvJob {
    using F = Fmt<FMT>;
    using XSrc = typename std::conditional<XSM, XSmem, XGlob>::type;
    struct Cursor {
        int row, blk, r0, r1, b0, b1, ks;
        bool valid;
    };
    // engine
    int nslots;
    uint32_t slot_bytes, job_smem_bytes;
    // problem
    const uint8_t *W, *Wend;
    int N, K, M, nbr, KS, groups, R, segb;  // segb == 0: whole rows per stage
    uint32_t rb;
    const float *x;                         // XSM: fp32 activations (M x K)
    const int8_t *xq;                       // !XSM: quantized activations
    const float *xd;
    const int32_t *xs;
    float *out;                             // y (KS == 1) or partials [KS][M][N]
    long slice_stride;
    uint32_t x_off;                         // XSM: offset of the x area in job smem
    int kslice_max;                         // XSM: activation columns reserved per token

    __device__ void first(Cursor &c) const {
        c.ks = blockIdx.x % KS;
        const int g = blockIdx.x / KS;
        c.r0 = (int)((long)g * N / groups);
        c.r1 = (int)((long)(g + 1) * N / groups);
        c.b0 = (int)((long)c.ks * nbr / KS);
        c.b1 = (int)((long)(c.ks + 1) * nbr / KS);
        c.row = c.r0;
        c.blk = c.b0;
        c.valid = c.r0 < c.r1 && c.b0 < c.b1;
    }
    __device__ void next(Cursor &c) const {
        if (segb == 0) {
            c.row += R;
        } else {
            c.blk += segb;
            if (c.blk >= c.b1) {
                c.blk = c.b0;
                ++c.row;
            }
        }
        c.valid = c.row < c.r1;
    }
    __device__ void stage(const Cursor &c, uint8_t *, bool, Stage &st) const {
        if (segb == 0) {
            const int nr = min(R, c.r1 - c.row);
            st.src[0] = W + (size_t)c.row * rb;
            st.bytes[0] = (uint32_t)nr * rb;
            st.R = nr;
            st.nblk = nbr;
            st.xb0 = 0;
            st.tag1 = 1;
        } else {
            const int nb = min(segb, c.b1 - c.blk);
            st.src[0] = W + (size_t)c.row * rb + (size_t)c.blk * F::BS;
            st.bytes[0] = (uint32_t)(nb * F::BS);
            st.R = 1;
            st.nblk = nb;
            st.xb0 = (XSM ? (c.blk - c.b0) : c.blk) * F::UPB;
            st.tag1 = (c.blk + nb >= c.b1);
        }
        st.src[1] = st.src[0];
        st.lim[0] = st.lim[1] = Wend;
        st.bytes[1] = 0;
        st.nseg = 1;
        st.rstride = rb;
        st.xm = 0;
        st.ntok = M;
        st.tag0 = c.row;
        st.tag2 = c.ks;
    }
    __device__ XSrc xsrc(uint8_t *, uint32_t job_base) const {
        if constexpr (XSM) {
            const XArea a = make_xarea(job_base + x_off, M, kslice_max);
            return XSmem{a.q, a.d, a.s, a.ldq, a.lds};
        } else {
            return XGlob{xq, xd, xs, K, K / 32};
        }
    }
    __device__ void producer_prologue(uint8_t *, int) const {}
    __device__ void consumer_prologue(uint8_t *js, int tid) const {
        float *racc = reinterpret_cast<float *>(js);
        if (tid < 16) racc[tid] = 0.0f;
        if constexpr (XSM) {
            Cursor c;
            first(c);
            if (!c.valid) return;
            const int c0 = c.b0 * F::QK, cols = (c.b1 - c.b0) * F::QK;
            const uint32_t base = smem_addr(js) + x_off;
            const XArea a = make_xarea(base, M, kslice_max);
            quantize_rows_to_smem(x + c0, K, M, cols, a.q, a.d, a.s, a.ldq, a.lds, tid, nullptr, nullptr,
                                  nullptr);
        }
    }
    template <int MT>
    __device__ void epilogue(const Stage &st, float *part, uint8_t *js, int tid) const {
        float *o = out + (long)st.tag2 * slice_stride;
        if (segb == 0) {
            for (int idx = tid; idx < st.R * M; idx += NCONS) {
                const int i = idx / M, m = idx - i * M;
                o[(long)m * N + st.tag0 + i] = part_take<MT>(part, i, m);
            }
        } else if (tid < M) {
            float *racc = reinterpret_cast<float *>(js);
            const float v = racc[tid] + part_take<MT>(part, 0, tid);
            if (st.tag1) {
                o[(long)tid * N + st.tag0] = v;
                racc[tid] = 0.0f;
            } else {
                racc[tid] = v;
            }
        }
    }
};

// ===================================================================================== FFN gate/up
template <int FMT, bool XSM>
struct FfnGateUpJob {
    using F = Fmt<FMT>;
    using XSrc = typename std::conditional<XSM, XSmem, XGlob>::type;
    struct Cursor {
        int row, r1;
        bool valid;
    };
    int nslots;
    uint32_t slot_bytes, job_smem_bytes;
    const uint8_t *Wg, *Wu, *Wg_end, *Wu_end;
    int H, I, M, nbr, R;
    uint32_t rb;
    const float *x;
    const int8_t *xq;
    const float *xd;
    const int32_t *xs;
    float *g_out, *u_out, *h_out;  // M x I
    uint32_t x_off;

    __device__ void first(Cursor &c) const {
        c.row = (int)((long)blockIdx.x * I / gridDim.x);
        c.r1 = (int)((long)(blockIdx.x + 1) * I / gridDim.x);
        c.valid = c.row < c.r1;
    }
    __device__ void next(Cursor &c) const {
        c.row += R;
        c.valid = c.row < c.r1;
    }
    __device__ void stage(const Cursor &c, uint8_t *, bool, Stage &st) const {
        const int nr = min(R, c.r1 - c.row);
        st.src[0] = Wg + (size_t)c.row * rb;
        st.src[1] = Wu + (size_t)c.row * rb;
        st.lim[0] = Wg_end;
        st.lim[1] = Wu_end;
        st.bytes[0] = st.bytes[1] = (uint32_t)nr * rb;
        st.nseg = 2;
        st.R = nr;
        st.rstride = rb;
        st.nblk = nbr;
        st.xb0 = 0;
        st.xm = 0;
        st.ntok = M;
        st.tag0 = c.row;
        st.tag1 = st.tag2 = 0;
    }
    __device__ XSrc xsrc(uint8_t *, uint32_t job_base) const {
        if constexpr (XSM) {
            const XArea a = make_xarea(job_base + x_off, M, H);
            return XSmem{a.q, a.d, a.s, a.ldq, a.lds};
        } else {
            return XGlob{xq, xd, xs, H, H / 32};
        }
    }
    __device__ void producer_prologue(uint8_t *, int) const {}
    __device__ void consumer_prologue(uint8_t *js, int tid) const {
        if constexpr (XSM) {
            const XArea a = make_xarea(smem_addr(js) + x_off, M, H);
            quantize_rows_to_smem(x, H, M, H, a.q, a.d, a.s, a.ldq, a.lds, tid, nullptr, nullptr, nullptr);
        }
    }
    template <int MT>
    __device__ void epilogue(const Stage &st, float *part, uint8_t *, int tid) const {
        for (int idx = tid; idx < st.R * M; idx += NCONS) {
            const int i = idx / M, m = idx - i * M;
            const float g = part_take<MT>(part, i, m);
            const float u = part_take<MT>(part, st.R + i, m);
            const long o = (long)m * I + st.tag0 + i;
            g_out[o] = g;
            u_out[o] = u;
            h_out[o] = silu_mul(g, u);
        }
    }
};

// ===================================================================================== MoE gate/up
constexpr int TOPK_MAX = 16;
constexpr int E_MAX = 1024;

template <int FMT, bool XSM>
struct MoeGateUpJob {
    using F = Fmt<FMT>;
    using XSrc = typename std::conditional<XSM, XSmem, XGlob>::type;
    struct Cursor {
        long p, p1;
        bool valid;
    };
    int nslots;
    uint32_t slot_bytes, job_smem_bytes;
    const uint8_t *Wg_exps, *Wu_exps, *Wg_sh, *Wu_sh;
    const uint8_t *Wg_exps_end, *Wu_exps_end, *Wg_sh_end, *Wu_sh_end;
    int E, topk, H, I, M, nbr, R;
    uint32_t rb;
    size_t ebytes;               // bytes of one expert matrix
    const float *logits;         // M x E
    int32_t *ids_ws;             // M x topk (always written)
    float *w_ws;
    int32_t *ids_out;            // nullable
    float *w_out;
    const float *x;
    const int8_t *xq;
    const float *xd;
    const int32_t *xs;
    float *g_out, *u_out, *h_out;  // [M][topk+1][I]
    uint32_t x_off;                // job smem: [ids M*topk int32][x area]

    __device__ int slots() const { return topk + 1; }
    __device__ void first(Cursor &c) const {
        const long P = (long)M * slots() * I;
        c.p = P * blockIdx.x / gridDim.x;
        c.p1 = P * (blockIdx.x + 1) / gridDim.x;
        c.valid = c.p < c.p1;
    }
    __device__ int rows_of(const Cursor &c) const {
        const int j = (int)(c.p % I);
        return (int)min((long)R, min(c.p1 - c.p, (long)(I - j)));
    }
    __device__ void next(Cursor &c) const {
        c.p += rows_of(c);
        c.valid = c.p < c.p1;
    }
    __device__ void stage(const Cursor &c, uint8_t *js, bool producer, Stage &st) const {
        const int gs = (int)(c.p / I), j = (int)(c.p % I);
        const int nr = rows_of(c);
        const int m = gs / slots(), s = gs - m * slots();
        st.src[0] = st.src[1] = nullptr;
        st.lim[0] = st.lim[1] = nullptr;
        if (producer) {
            const int32_t *ids = reinterpret_cast<const int32_t *>(js);
            if (s < topk) {
                const size_t e = (size_t)min(max(ids[m * topk + s], 0), E - 1);  // never leave the tensor
                st.src[0] = Wg_exps + e * ebytes + (size_t)j * rb;
                st.src[1] = Wu_exps + e * ebytes + (size_t)j * rb;
                st.lim[0] = Wg_exps_end;
                st.lim[1] = Wu_exps_end;
            } else {
                st.src[0] = Wg_sh + (size_t)j * rb;
                st.src[1] = Wu_sh + (size_t)j * rb;
                st.lim[0] = Wg_sh_end;
                st.lim[1] = Wu_sh_end;
            }
        }
        st.bytes[0] = st.bytes[1] = (uint32_t)nr * rb;
        st.nseg = 2;
        st.R = nr;
        st.rstride = rb;
        st.nblk = nbr;
        st.xb0 = 0;
        st.xm = m;
        st.ntok = 1;
        st.tag0 = gs;
        st.tag1 = j;
        st.tag2 = 0;
    }
    __device__ XSrc xsrc(uint8_t *, uint32_t job_base) const {
        if constexpr (XSM) {
            const XArea a = make_xarea(job_base + x_off, M, H);
            return XSmem{a.q, a.d, a.s, a.ldq, a.lds};
        } else {
            return XGlob{xq, xd, xs, H, H / 32};
        }
    }
    // Router tail, one warp: softmax over E logits, the topk largest (ties: lower id),
    // weights renormalized over the picks.  exp(l - max) / sum over the picks equals
    // p / sum(p over the picks) for the softmax probabilities p.
    __device__ void producer_prologue(uint8_t *js, int lane) const {
        int32_t *ids = reinterpret_cast<int32_t *>(js);
        for (int m = 0; m < M; ++m) {
            float v[E_MAX / 32];
            float lmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < E_MAX / 32; ++i) {
                const int e = lane + 32 * i;
                v[i] = e < E ? logits[(long)m * E + e] : -INFINITY;
                lmax = fmaxf(lmax, v[i]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
            uint32_t taken = 0;
            int sel[TOPK_MAX];
            float ev[TOPK_MAX];
            float esum = 0.0f;
#pragma unroll
            for (int r = 0; r < TOPK_MAX; ++r) {
                sel[r] = 0;
                ev[r] = 0.0f;
                if (r < topk) {
                    float bv = -INFINITY;
                    int be = 0x7fffffff;
#pragma unroll
                    for (int i = 0; i < E_MAX / 32; ++i) {
                        const int e = lane + 32 * i;
                        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || be == 0x7fffffff)) {
                            bv = v[i];
                            be = e;
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                        if (ov > bv || (ov == bv && oe < be)) {
                            bv = ov;
                            be = oe;
                        }
                    }
                    if ((be & 31) == lane) taken |= 1u << (be >> 5);
                    sel[r] = be;
                    ev[r] = expf(bv - lmax);
                    esum += ev[r];
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < TOPK_MAX; ++r) {
                    if (r < topk) {
                        const float w = ev[r] / esum;
                        ids[m * topk + r] = sel[r];
                        if (blockIdx.x == 0) {
                            ids_ws[m * topk + r] = sel[r];
                            w_ws[m * topk + r] = w;
                            if (ids_out) ids_out[m * topk + r] = sel[r];
                            if (w_out) w_out[m * topk + r] = w;
                        }
                    }
                }
            }
            __syncwarp();
        }
    }
    __device__ void consumer_prologue(uint8_t *js, int tid) const {
        if constexpr (XSM) {
            const XArea a = make_xarea(smem_addr(js) + x_off, M, H);
            quantize_rows_to_smem(x, H, M, H, a.q, a.d, a.s, a.ldq, a.lds, tid, nullptr, nullptr, nullptr);
        }
    }
    template <int MT>
    __device__ void epilogue(const Stage &st, float *part, uint8_t *, int tid) const {
        for (int i = tid; i < st.R; i += NCONS) {
            const float g = part_take<MT>(part, i, 0);
            const float u = part_take<MT>(part, st.R + i, 0);
            const long o = (long)st.tag0 * I + st.tag1 + i;
            g_out[o] = g;
            u_out[o] = u;
            h_out[o] = silu_mul(g, u);
        }
    }
};

// ===================================================================================== MoE down
template <int FMT, bool XSM>
struct MoeDownJob {
    using F = Fmt<FMT>;
    using XSrc = typename std::conditional<XSM, XSmem, XGlob>::type;
    struct Cursor {
        int m, s, n, n0, n1;
        bool valid;
    };
    int nslots;
    uint32_t slot_bytes, job_smem_bytes;
    const uint8_t *Wd_exps, *Wd_sh, *Wd_exps_end, *Wd_sh_end;
    int E, topk, H, I, M, nbr, R, nloc_max;
    uint32_t rb;
    size_t ebytes;
    const int32_t *ids_ws;
    const float *w_ws;
    const float *h;                 // [M][S][I] fp32 (XSM: quantized here)
    const int8_t *hq;               // !XSM: requantized h in global memory
    const float *hd;
    const int32_t *hs;
    int8_t *hq_ws;                  // XSM: CTA 0 mirrors its requantization here
    float *hd_ws;
    int32_t *hs_ws;
    float *y;                       // M x H
    uint32_t x_off;                 // job smem: [yacc M*nloc_max fp32][x area]

    __device__ int slots() const { return topk + 1; }
    __device__ void first(Cursor &c) const {
        c.n0 = (int)((long)blockIdx.x * H / gridDim.x);
        c.n1 = (int)((long)(blockIdx.x + 1) * H / gridDim.x);
        c.m = 0;
        c.s = 0;
        c.n = c.n0;
        c.valid = c.n0 < c.n1;
    }
    __device__ void next(Cursor &c) const {
        c.n += R;
        if (c.n >= c.n1) {
            c.n = c.n0;
            if (++c.s == slots()) {
                c.s = 0;
                ++c.m;
            }
        }
        c.valid = c.m < M;
    }
    __device__ void stage(const Cursor &c, uint8_t *, bool producer, Stage &st) const {
        const int nr = min(R, c.n1 - c.n);
        st.src[0] = st.src[1] = nullptr;
        st.lim[0] = st.lim[1] = nullptr;
        if (producer) {
            if (c.s < topk) {
                const size_t e = (size_t)min(max(ids_ws[c.m * topk + c.s], 0), E - 1);
                st.src[0] = Wd_exps + e * ebytes + (size_t)c.n * rb;
                st.lim[0] = Wd_exps_end;
            } else {
                st.src[0] = Wd_sh + (size_t)c.n * rb;
                st.lim[0] = Wd_sh_end;
            }
            st.src[1] = st.src[0];
            st.lim[1] = st.lim[0];
        }
        st.bytes[0] = (uint32_t)nr * rb;
        st.bytes[1] = 0;
        st.nseg = 1;
        st.R = nr;
        st.rstride = rb;
        st.nblk = nbr;
        st.xb0 = 0;
        st.xm = c.m * slots() + c.s;
        st.ntok = 1;
        st.tag0 = c.m;
        st.tag1 = c.s;
        st.tag2 = c.n - c.n0;
    }
    __device__ XSrc xsrc(uint8_t *, uint32_t job_base) const {
        if constexpr (XSM) {
            const XArea a = make_xarea(job_base + x_off, M * (topk + 1), I);
            return XSmem{a.q, a.d, a.s, a.ldq, a.lds};
        } else {
            return XGlob{hq, hd, hs, I, I / 32};
        }
    }
    __device__ void producer_prologue(uint8_t *, int) const {}
    __device__ void consumer_prologue(uint8_t *js, int tid) const {
        float *yacc = reinterpret_cast<float *>(js);
        for (int i = tid; i < M * nloc_max; i += NCONS) yacc[i] = 0.0f;
        if constexpr (XSM) {
            const int rows = M * (topk + 1);
            const XArea a = make_xarea(smem_addr(js) + x_off, rows, I);
            const bool mirror = blockIdx.x == 0;
            quantize_rows_to_smem(h, I, rows, I, a.q, a.d, a.s, a.ldq, a.lds, tid, mirror ? hq_ws : nullptr,
                                  mirror ? hd_ws : nullptr, mirror ? hs_ws : nullptr);
        }
    }
    template <int MT>
    __device__ void epilogue(const Stage &st, float *part, uint8_t *js, int tid) const {
        float *yacc = reinterpret_cast<float *>(js);
        const int m = st.tag0, s = st.tag1;
        const float wgt = s < topk ? w_ws[m * topk + s] : 1.0f;  // shared expert: weight 1
        for (int i = tid; i < st.R; i += NCONS) {
            const float o = part_take<MT>(part, i, 0);
            float *a = yacc + m * nloc_max + st.tag2 + i;
            const float v = fmaf(wgt, o, *a);
            if (s == topk) {
                Cursor c;
                first(c);
                y[(long)m * H + c.n0 + st.tag2 + i] = v;
            } else {
                *a = v;
            }
        }
    }
};

}  // namespace qg
