// qg_jobs.cuh -- the four GEMV-shaped operations as output-row jobs for the streaming
// engine (qg_engine.cuh):
//
//   GemvJob        output row n = row n of W (optionally one K-slice per CTA: split-K,
//                  partial sums to a buffer)
//   FfnGateUpJob   output rows 0..I-1 = rows of Wg (g), I..2I-1 = rows of Wu (u)
//   MoeGateUpJob   output rows of g and u for every (token, slot): the slot's routed expert
//                  (from the router's top-k, computed in the prologue) or the shared one;
//                  each CTA owns whole 32-blocks of positions and its epilogue requantizes
//                  h = silu(g) * u into the down projection's activation tiles
//   MoeDownJob     per CTA, a range of hidden rows n: output rows (token, slot, n) of every
//                  slot's down matrix, kept in shared memory; the epilogue forms
//                  y[token][n] = sum over slots, in slot order, of weight * row (shared
//                  expert: weight 1) -- the weighted aggregation of the expert outputs
//
// Engine interface: HAS_FINISH, HAS_PROLOGUE; fields depth, slot_bytes, x_bytes, j_bytes,
// tpr_x, tps, ntok; Ctx ctx() (per-CTA constants, computed once and passed to the calls
// below); cta(o0, o1, tpr, grp), seg_src, xrows/xrow_src/xrow_bytes, xrow, store, init,
// finish, prologue (run by every warp before any weight copy, e.g. the MoE top-k).
// The engine may start before the previous kernel in the stream has finished (programmatic
// dependent launch): seg_src may only read data no earlier kernel writes (the weights),
// unless the job's prologue first waits for the previous kernel (griddep_wait).
// Activation images (prep_tiles_warp) have one row of task tiles per token (or per MoE
// slot), row pitch tpr * tile_stride(XGT).  The MoE jobs take P activation rows per token
// (or slot): P = 2 for s16 activations held as two int8 planes (prep_tiles_s16_warp); the
// engine then runs P tokens per lane over one row's planes, and the P results of an output
// row are kept apart for the next step to add.
#pragma once

#include "qg_engine.cuh"

namespace qg {

struct EngineFields {
    int depth;                          // ring slots per consumer warp
    uint32_t slot_bytes, x_bytes, j_bytes;
    int tpr_x, tps, ntok;
    int xrep;  // activation tiles repeated past a row's end (virtual columns), 0 = none
};

// ===================================================================================== GEMV
template <int FMT, int T>
struct GemvJob : EngineFields {
    using F = FT<FMT, T>;
    static constexpr bool HAS_FINISH = false, HAS_PROLOGUE = false;
    const uint8_t *W, *Wend;
    int N, KS, groups, gpr;  // gpr: task groups (whole blocks) per row
    uint32_t rb;
    const uint8_t *ximg;
    uint32_t ximg_pitch;
    float *out;  // y (KS == 1) or partials [KS][M][N]
    long slice_stride;

    // per-CTA constants: K-slice, its first task, its tasks per row, the output slice
    struct Ctx {
        int ks, t0, tpr, o0, o1;
        float *out;
    };
    __device__ Ctx ctx() const {
        Ctx c;
        const int g = KS == 1 ? (int)blockIdx.x : (int)blockIdx.x / KS;
        c.ks = KS == 1 ? 0 : (int)blockIdx.x - g * KS;
        c.t0 = split_point(gpr, c.ks, KS) * F::TPB;
        c.tpr = split_point(gpr, c.ks + 1, KS) * F::TPB - c.t0;
        c.o0 = split_point(N, g, groups);
        c.o1 = split_point(N, g + 1, groups);
        c.out = out + (long)c.ks * slice_stride;
        return c;
    }
    __device__ void cta(const Ctx &c, int &o0, int &o1, int &tpr, int &grp) const {
        o0 = c.o0;
        o1 = c.o1;
        tpr = c.tpr;
        grp = KS == 1 ? 0 : 1;  // slices of consecutive rows are not adjacent
    }
    __device__ const uint8_t *seg_src(const Ctx &c, int o, int tt, const uint8_t *&lim, const int *) const {
        lim = Wend;
        return W + (size_t)o * rb + task_off<F>(c.t0 + tt);
    }
    __device__ int xrows() const { return ntok; }
    __device__ const uint8_t *xrow_src(const Ctx &c, int r) const {
        return ximg + (size_t)r * ximg_pitch + (size_t)c.t0 * tile_stride(F::XGT);
    }
    __device__ uint32_t xrow_bytes(const Ctx &c, int) const { return (uint32_t)(c.tpr * tile_stride(F::XGT)); }
    __device__ uint32_t xrow(const Ctx &, int, const FastDiv &) const { return 0; }
    __device__ void store(const Ctx &c, int o, int m, float v, float *) const { c.out[(long)m * N + o] = v; }
    __device__ void init(float *, int) const {}
    __device__ void finish(const Ctx &, float *, int, int, const int *) const {}
    __device__ void prologue(int, int, int, int *) const {}
};

// ===================================================================================== FFN gate/up
template <int FMT, int T>
struct FfnGateUpJob : EngineFields {
    using F = FT<FMT, T>;
    static constexpr bool HAS_FINISH = false, HAS_PROLOGUE = false;
    const uint8_t *Wg, *Wu, *Wg_end, *Wu_end;
    int I, m0;  // tokens [m0, m0 + ntok) of the batch
    uint32_t rb;
    const uint8_t *ximg;
    uint32_t ximg_pitch;
    float *g_out, *u_out;  // row pitch I, whole batch

    struct Ctx {};
    __device__ Ctx ctx() const { return {}; }
    __device__ void cta(const Ctx &, int &o0, int &o1, int &tpr, int &grp) const {
        o0 = split_point(2L * I, (int)blockIdx.x, (int)gridDim.x);
        o1 = split_point(2L * I, (int)blockIdx.x + 1, (int)gridDim.x);
        tpr = tpr_x;
        grp = I;
    }
    __device__ const uint8_t *seg_src(const Ctx &, int o, int tt, const uint8_t *&lim, const int *) const {
        const bool up = o >= I;
        lim = up ? Wu_end : Wg_end;
        return (up ? Wu : Wg) + (size_t)(up ? o - I : o) * rb + task_off<F>(tt);
    }
    __device__ int xrows() const { return ntok; }
    __device__ const uint8_t *xrow_src(const Ctx &, int r) const { return ximg + (size_t)(m0 + r) * ximg_pitch; }
    __device__ uint32_t xrow_bytes(const Ctx &, int) const { return ximg_pitch; }
    __device__ uint32_t xrow(const Ctx &, int, const FastDiv &) const { return 0; }
    __device__ void store(const Ctx &, int o, int m, float v, float *) const {
        if (o < I)
            g_out[(long)(m0 + m) * I + o] = v;
        else
            u_out[(long)(m0 + m) * I + o - I] = v;
    }
    __device__ void init(float *, int) const {}
    __device__ void finish(const Ctx &, float *, int, int, const int *) const {}
    __device__ void prologue(int, int, int, int *) const {}
};

// ===================================================================================== MoE gate/up
constexpr int TOPK_MAX = 16;
constexpr int E_MAX = 1024;

template <int FMT, int T, int P = 1>
struct MoeGateUpJob : EngineFields {
    using F = FT<FMT, T>;
    static constexpr bool HAS_FINISH = true, HAS_PROLOGUE = true;
    const uint8_t *Wg_exps, *Wu_exps, *Wg_sh, *Wu_sh;
    const uint8_t *Wg_exps_end, *Wu_exps_end, *Wg_sh_end, *Wu_sh_end;
    int E, topk, I, M;
    int nunits;                  // M * (topk + 1) * I / 32 units of 32 positions j
    FastDiv div_slots;           // by topk + 1
    FastDiv div_ub;              // by I / 32
    uint32_t rb;
    size_t ebytes;               // bytes of one expert matrix
    const float *logits;         // M x E (written by the previous kernel)
    int32_t *ids_ws;             // M x topk (always written)
    float *w_ws;
    int32_t *ids_out;            // nullable
    float *w_out;
    const uint8_t *ximg;         // P rows per token
    uint32_t ximg_pitch;
    float *g_out, *u_out;        // [M][topk+1][P][I]
    // h = silu(g) * u requantized (int8, or s16 as two planes): the down projection's
    // activation tile image (P rows per (token, slot), tiles of 2^himg_xgt_log2 blocks,
    // himg_tpr tasks per row), and the plain h, codes (int8 or int16), steps and code sums
    uint8_t *himg;
    int himg_tpr, himg_xgt_log2;
    float *h_out;
    void *hq;
    float *hd;
    int32_t *hs;

    __device__ int slots() const { return topk + 1; }
    // The CTA owns units [u0, u0 + nu); unit (token * slots + slot) * I/32 + jb holds the
    // gate and up rows j = 32 jb .. 32 jb + 31 of that slot's expert, so that the CTA can
    // requantize whole 32-blocks of h when its rows are done.  CTA-local rows:
    // o = 64 * (unit - u0) + 32 * up + (j & 31); runs of 32 adjacent rows.
    struct Ctx {
        int u0, nu;
    };
    __device__ Ctx ctx() const {
        Ctx c;
        c.u0 = split_point(nunits, (int)blockIdx.x, (int)gridDim.x);
        c.nu = split_point(nunits, (int)blockIdx.x + 1, (int)gridDim.x) - c.u0;
        return c;
    }
    __device__ void cta(const Ctx &c, int &o0, int &o1, int &tpr, int &grp) const {
        o0 = 0;
        o1 = 64 * c.nu;
        tpr = tpr_x;
        grp = 32;
    }
    // (token * slots + slot, jb) of CTA-local row o
    __device__ __forceinline__ int unit_gs(const Ctx &c, int o, int &jb) const {
        const int un = c.u0 + (o >> 6);
        const int gs = (int)div_ub.div((uint32_t)un);
        jb = un - gs * (I >> 5);
        return gs;
    }
    __device__ const uint8_t *seg_src(const Ctx &c, int o, int tt, const uint8_t *&lim, const int *ids) const {
        int jb;
        const int gs = unit_gs(c, o, jb), up = (o >> 5) & 1, j = 32 * jb + (o & 31);
        const int m = (int)div_slots.div((uint32_t)gs), s = gs - m * slots();
        if (s < topk) {
            const size_t e = (size_t)min(max(ids[m * topk + s], 0), E - 1);  // never leave the tensor
            lim = up ? Wu_exps_end : Wg_exps_end;
            return (up ? Wu_exps : Wg_exps) + e * ebytes + (size_t)j * rb + task_off<F>(tt);
        }
        lim = up ? Wu_sh_end : Wg_sh_end;
        return (up ? Wu_sh : Wg_sh) + (size_t)j * rb + task_off<F>(tt);
    }
    __device__ int xrows() const { return M * P; }
    __device__ const uint8_t *xrow_src(const Ctx &, int r) const { return ximg + (size_t)r * ximg_pitch; }
    __device__ uint32_t xrow_bytes(const Ctx &, int) const { return ximg_pitch; }
    __device__ uint32_t xrow(const Ctx &c, int o, const FastDiv &) const {
        int jb;
        return P * div_slots.div((uint32_t)unit_gs(c, o, jb));  // the token's first row
    }
    // g or u of plane m to the workspace and to the CTA's job area (64 * nu * P floats)
    __device__ void store(const Ctx &c, int o, int m, float v, float *part) const {
        int jb;
        const int gs = unit_gs(c, o, jb), j = 32 * jb + (o & 31);
        (((o >> 5) & 1) ? u_out : g_out)[((long)gs * P + m) * I + j] = v;
        part[o * P + m] = v;
    }
    __device__ void init(float *, int) const {}
    // One warp per unit: h = silu(g) * u for its 32 positions (g, u: the planes' partial
    // rows added in plane order), quantized by the activation rule of the call and written
    // into the down projection's tile image and the workspace.
    __device__ void finish(const Ctx &c, float *part, int tid, int nthreads, const int *scratch) const {
        const int lane = tid & 31;
        for (int i = tid >> 5; i < c.nu; i += nthreads >> 5) {
            int jb;
            const int gs = unit_gs(c, 64 * i, jb);
            const float *pg = part + (64 * i + lane) * P, *pu = part + (64 * i + 32 + lane) * P;
            float g = pg[0], u = pu[0];
#pragma unroll
            for (int p = 1; p < P; ++p) {
                g += pg[p];
                u += pu[p];
            }
            const float h = silu_mul(g, u);
            const long e = (long)gs * I + 32 * jb + lane, eb = (long)gs * (I >> 5) + jb;
            h_out[e] = h;
            int q, sum;
            float d;
            if constexpr (P == 2) {
                quant_block_warp16(h, q, d, sum);
                put_block_s16(himg, gs, himg_tpr, jb, himg_xgt_log2, lane, q, d, sum);
                static_cast<int16_t *>(hq)[e] = (int16_t)q;
            } else {
                quant_block_warp(h, q, d, sum);
                put_block(himg, gs, himg_tpr, jb, himg_xgt_log2, lane, q, d, sum);
                static_cast<int8_t *>(hq)[e] = (int8_t)q;
            }
            if (lane == 0) {
                hd[eb] = d;
                hs[eb] = sum;
            }
        }
    }
    // Router tail, after the logits kernel has finished: softmax over E logits, the topk
    // largest (ties: lower id), weights renormalized over the picks; one warp per token.
    // exp(l - max) / sum over the picks equals p / sum(p over the picks) for the softmax
    // probabilities p; the sum runs over the picks in pick order.
    __device__ void prologue(int warp, int nwarps, int lane, int *ids) const {
        griddep_wait();
        if (E <= 256 && topk <= 8)
            select_topk8(warp, nwarps, lane, ids);
        else if (E <= 256)
            select_topk<256 / 32>(warp, nwarps, lane, ids);
        else
            select_topk<E_MAX / 32>(warp, nwarps, lane, ids);
    }
    // Pick order as one 64-bit key: the logit's order-preserving bits above, the complement
    // of the expert id below (so that of equal logits the lower id ranks higher).
    __device__ static __forceinline__ uint64_t pick_key(float v, int e) {
        const uint32_t b = __float_as_uint(v);
        const uint32_t u = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        return ((uint64_t)u << 32) | (uint64_t)(0xffffffffu - (uint32_t)e);
    }
    __device__ static __forceinline__ float pick_value(uint64_t k) {
        const uint32_t u = (uint32_t)(k >> 32);
        return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
    }
    __device__ static __forceinline__ int pick_id(uint64_t k) { return (int)(0xffffffffu - (uint32_t)k); }
    __device__ static __forceinline__ void cas_desc(uint64_t &a, uint64_t &b) {
        const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
        a = hi;
        b = lo;
    }
    // E <= 256, topk <= 8.  Each lane sorts the keys of its 8 logits (a 19-comparator
    // network), then five butterfly rounds merge the lists of lane pairs keeping the best 8
    // (the larger of a[i] and b[7 - i] form a bitonic sequence holding the 8 best of both
    // lists, sorted by three rounds of compare-exchanges); every lane ends with the row's 8
    // best keys in pick order.  The keys are distinct, so the picks, their order and the
    // weights are those of taking the largest remaining logit topk times.
    __device__ void select_topk8(int warp, int nwarps, int lane, int *ids) const {
        for (int m = warp; m < M; m += nwarps) {
            uint64_t c[8];
            float lmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                const float v = e < E ? logits[(long)m * E + e] + 0.0f : -INFINITY;  // + 0: -0 as +0
                lmax = fmaxf(lmax, v);
                c[i] = e < E ? pick_key(v, e) : 0ull;  // 0: below every logit's key
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
            cas_desc(c[0], c[2]); cas_desc(c[1], c[3]); cas_desc(c[4], c[6]); cas_desc(c[5], c[7]);
            cas_desc(c[0], c[4]); cas_desc(c[1], c[5]); cas_desc(c[2], c[6]); cas_desc(c[3], c[7]);
            cas_desc(c[0], c[1]); cas_desc(c[2], c[3]); cas_desc(c[4], c[5]); cas_desc(c[6], c[7]);
            cas_desc(c[2], c[4]); cas_desc(c[3], c[5]);
            cas_desc(c[1], c[4]); cas_desc(c[3], c[6]);
            cas_desc(c[1], c[2]); cas_desc(c[3], c[4]); cas_desc(c[5], c[6]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                uint64_t b[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) b[i] = __shfl_xor_sync(0xffffffffu, c[i], o);
#pragma unroll
                for (int i = 0; i < 8; ++i) c[i] = c[i] > b[7 - i] ? c[i] : b[7 - i];
#pragma unroll
                for (int d = 4; d > 0; d >>= 1)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if ((i & d) == 0) cas_desc(c[i], c[i + d]);
            }
            float esum = 0.0f, my_ev = 0.0f;
            int my_sel = 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (r < topk) {
                    const float ev = expf(pick_value(c[r]) - lmax);
                    esum += ev;
                    if (lane == r) {
                        my_sel = pick_id(c[r]);
                        my_ev = ev;
                    }
                }
            }
            if (lane < topk) {
                const float w = my_ev / esum;
                ids[m * topk + lane] = my_sel;
                if (blockIdx.x == 0) {
                    ids_ws[m * topk + lane] = my_sel;
                    w_ws[m * topk + lane] = w;
                    if (ids_out) ids_out[m * topk + lane] = my_sel;
                    if (w_out) w_out[m * topk + lane] = w;
                }
            }
            __syncwarp();
        }
    }
    // General E and topk: a round of the selection is two warp reductions, the largest logit
    // (as an order-preserving integer key), then the lowest expert id holding it.  Each lane
    // keeps the best of its own NV logits; only the lane whose logit was taken rescans.
    template <int NV>
    __device__ void select_topk(int warp, int nwarps, int lane, int *ids) const {
        for (int m = warp; m < M; m += nwarps) {
            float v[NV];
            float lmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int e = lane + 32 * i;
                v[i] = e < E ? logits[(long)m * E + e] + 0.0f : -INFINITY;  // + 0: -0 as +0
                lmax = fmaxf(lmax, v[i]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
            uint32_t taken = 0;
            float bv;
            int be;
            // this lane's largest remaining logit (its lowest id on ties)
            auto rescan = [&]() {
                bv = -INFINITY;
                be = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && !((taken >> i) & 1u) && (v[i] > bv || be == 0x7fffffff)) {
                        bv = v[i];
                        be = e;
                    }
                }
            };
            rescan();
            float esum = 0.0f;
            int my_sel = 0;
            float my_ev = 0.0f;
            for (int r = 0; r < topk; ++r) {
                const int bits = __float_as_int(bv);
                const int key = be == 0x7fffffff ? (int)0x80000000 : (bits >= 0 ? bits : bits ^ 0x7fffffff);
                const int kmax = __reduce_max_sync(0xffffffffu, key);
                const int sel = __reduce_min_sync(0xffffffffu, key == kmax ? be : 0x7fffffff);
                const float sv = __int_as_float(kmax >= 0 ? kmax : kmax ^ 0x7fffffff);
                if ((sel & 31) == lane) {
                    taken |= 1u << (sel >> 5);
                    rescan();
                }
                const float ev = expf(sv - lmax);
                esum += ev;
                if (lane == r) {
                    my_sel = sel;
                    my_ev = ev;
                }
            }
            if (lane < topk) {
                const float w = my_ev / esum;
                ids[m * topk + lane] = my_sel;
                if (blockIdx.x == 0) {
                    ids_ws[m * topk + lane] = my_sel;
                    w_ws[m * topk + lane] = w;
                    if (ids_out) ids_out[m * topk + lane] = my_sel;
                    if (w_out) w_out[m * topk + lane] = w;
                }
            }
            __syncwarp();
        }
    }
};

// ===================================================================================== MoE down
template <int FMT, int T, int P = 1>
struct MoeDownJob : EngineFields {
    using F = FT<FMT, T>;
    static constexpr bool HAS_FINISH = true, HAS_PROLOGUE = true;
    const uint8_t *Wd_exps, *Wd_sh, *Wd_exps_end, *Wd_sh_end;
    int E, topk, H, M, m0;          // tokens [m0, m0 + M) of the batch
    uint32_t rb;
    size_t ebytes;
    const int32_t *ids_ws;          // [batch][topk] (written by the gate/up kernel)
    const float *w_ws;
    const uint8_t *ximg;            // requantized h: P image rows per (token, slot)
    uint32_t ximg_pitch;
    float *y;                       // [batch][H]

    __device__ int slots() const { return topk + 1; }
    // per-CTA constants: this CTA's hidden rows [n0, n0 + nloc) and the row decomposition
    struct Ctx {
        int n0, nloc;
        FastDiv dnloc, dslots;
    };
    __device__ Ctx ctx() const {
        Ctx c;
        c.n0 = split_point(H, (int)blockIdx.x, (int)gridDim.x);
        c.nloc = split_point(H, (int)blockIdx.x + 1, (int)gridDim.x) - c.n0;
        c.dnloc = FastDiv::make((uint32_t)c.nloc);
        c.dslots = FastDiv::make((uint32_t)slots());
        return c;
    }
    // CTA-local rows o = (token * slots + slot) * nloc + r, r < nloc
    __device__ void cta(const Ctx &c, int &o0, int &o1, int &tpr, int &grp) const {
        o0 = 0;
        o1 = M * slots() * c.nloc;
        tpr = tpr_x;
        grp = c.nloc;
    }
    __device__ const uint8_t *seg_src(const Ctx &c, int o, int tt, const uint8_t *&lim, const int *ids) const {
        const int q = (int)c.dnloc.div((uint32_t)o), r = o - q * c.nloc;
        const int m = (int)c.dslots.div((uint32_t)q), s = q - m * slots();
        if (s < topk) {
            const size_t e = (size_t)min(max(ids[m * topk + s], 0), E - 1);
            lim = Wd_exps_end;
            return Wd_exps + e * ebytes + (size_t)(c.n0 + r) * rb + task_off<F>(tt);
        }
        lim = Wd_sh_end;
        return Wd_sh + (size_t)(c.n0 + r) * rb + task_off<F>(tt);
    }
    __device__ int xrows() const { return M * slots() * P; }
    __device__ const uint8_t *xrow_src(const Ctx &, int r) const {
        return ximg + ((size_t)m0 * slots() * P + r) * ximg_pitch;
    }
    __device__ uint32_t xrow_bytes(const Ctx &, int) const { return ximg_pitch; }
    __device__ uint32_t xrow(const Ctx &, int o, const FastDiv &divn) const {
        return P * divn.div((uint32_t)o);  // first row of (token * slots + slot)
    }
    __device__ void store(const Ctx &, int o, int m, float v, float *part) const { part[o * P + m] = v; }
    __device__ void init(float *, int) const {}
    __device__ void finish(const Ctx &c, float *part, int tid, int nthreads, const int *scratch) const {
        const int nloc = c.nloc;
        for (int i = tid; i < M * nloc; i += nthreads) {
            const int m = i / nloc, r = i - m * nloc;
            float acc = 0.0f;
            for (int s = 0; s < slots(); ++s) {
                // shared expert: weight 1
                const float ws = s < topk ? __int_as_float(scratch[SCRATCH_W + m * topk + s]) : 1.0f;
                const float *o = part + ((m * slots() + s) * nloc + r) * P;
                float v = o[0];
#pragma unroll
                for (int p = 1; p < P; ++p) v += o[p];
                acc = fmaf(ws, v, acc);
            }
            y[(long)(m0 + m) * H + c.n0 + r] = acc;
        }
    }
    // The weight copies need the routed expert ids, written two kernels earlier: wait for
    // the previous kernel (and so for everything before it) before any copy is issued, then
    // bring this launch's ids and routing weights into shared memory (scratch[i] and
    // scratch[SCRATCH_W + i] for pick i of the launch's tokens).
    __device__ void prologue(int warp, int nwarps, int lane, int *scratch) const {
        griddep_wait();
        for (int i = warp * 32 + lane; i < M * topk; i += nwarps * 32) {
            scratch[i] = ids_ws[m0 * topk + i];
            scratch[SCRATCH_W + i] = __float_as_int(w_ws[m0 * topk + i]);
        }
    }
};

}  // namespace qg
