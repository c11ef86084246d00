// qg_engine1.cuh -- the one-token GEMV engine for rows that start 16-byte aligned.
//
// One token, one matrix, no K-split: a CTA owns the contiguous output rows [o0, o1), and
// because every row is tpr tasks of TASK_BYTES bytes laid out back to back, the CTA's tasks
// are one contiguous byte range: task f of the CTA starts at W + o0 * rb + f * TASK_BYTES.
// With TASK_BYTES and rb multiples of 16 every stage is then a single aligned bulk copy, and
// the bookkeeping of the general engine (run tables, widened pieces, segmented reductions
// with carries across stages and warps) is not needed:
//  * the CTA's tasks are split into NCW contiguous ranges, one per warp; a warp consumes its
//    range in stages of 32 tasks (lane l takes task 32 s + l) through D ring slots of its
//    own, lane 0 issuing one cp.async.bulk per stage, completion counted on the slot's
//    mbarrier;
//  * a lane copies its task from the slot into registers, the warp refills the slot with
//    the stage D ahead, and the lane decodes its task against the activation tiles (written
//    by the preparation kernel, copied once into shared memory, with the first 31 tiles
//    repeated after the row so that the 32 lanes of a stage read consecutive tiles even
//    where the stage wraps into the next row);
//  * each task's fp32 sum goes to part[row][task] in shared memory; after the last stage
//    the CTA adds every row's tpr partial sums in task order and writes y.  The order of
//    every addition is fixed, so results are deterministic.
#pragma once

#include "qg_engine.cuh"

namespace qg {

struct Gemv1Args {
    const uint8_t *W;      // N rows of rb bytes
    float *y;              // N outputs (one token)
    const uint8_t *ximg;   // activation tile image of the token's row: tpr tiles
    const float *x;        // or (non-null): the fp32 row of K elements, quantized by every CTA
    int N, K, tpr, depth, xrep;
    uint32_t rb, slot_bytes, x_bytes;
    int ra, nra;           // CTA row ranges start at multiples of ra rows (ra * rb: 16-byte multiple); nra = N / ra
};

// Tiles tpr .. tpr + xrep - 1 of a row image in shared memory (16-byte aligned) as copies
// of tiles (j mod tpr), in 16-byte chunks spread over nth threads.
template <int STRIDE>
__device__ __forceinline__ void repeat_tiles(uint8_t *xs, int tpr, int xrep, int tid, int nth) {
    constexpr int CPT = STRIDE / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(xs);
    uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)tpr * STRIDE);
    for (int c = tid; c < xrep * CPT; c += nth) {
        const int j = c / CPT;
        dst[c] = src[(j % tpr) * CPT + (c - j * CPT)];
    }
}

// The activation row x (K fp32 elements, 16-byte aligned) quantized by the NTH threads of a
// CTA straight into the shared tile image xs: tpr tiles of XGT blocks, the first xrep tiles
// repeated after the row, each unit laid out as put_tile_unit writes it.  The rule is
// quant_block_warp's (d = amax / 127 rounded to nearest, q = round(v / d) clamped to
// +-127, v / d the rounded quotient), taken by eight lanes per 32-element block, four
// elements each: the block's maximum and code sums are exact in any order, so the tiles
// equal those of the preparation kernel bit for bit.  A thread takes XCH blocks at a time
// side by side (their loads, reductions and divisions interleave), and v / d goes through
// the rounded reciprocal: |v * inv - fl(v / d)| < 2e-5 for |v| <= amax (both lie within a
// few 2^-24 relative of v / d <= 127), so rounding it gives round(fl(v / d)) unless it lies
// within 2^-14 of a half-integer; there, and for a subnormal d (no finite reciprocal), the
// rounded division decides.  The blocks are written once; the repeated tiles are copied
// from them after a barrier of the CTA (every thread calls this).  The row is read from L2 (it may have been written by the
// previous kernel).  after_loads() runs once, right after the first loads.
template <int XGT, int NTH, class AfterLoads>
__device__ __forceinline__ void quant_row_tiles(const float *x, int K, uint8_t *xs, int tpr, int xrep, int tid,
                                                AfterLoads &&after_loads) {
    constexpr int XCH = 4, NG = NTH / 8, STRIDE = tile_stride(XGT);
    const int nb = K / 32, grp = tid >> 3, sub = tid & 7;
    for (int b0 = 0; b0 < nb; b0 += NG * XCH) {
        float e[XCH][4];
#pragma unroll
        for (int i = 0; i < XCH; ++i) {
            const int b = b0 + grp + i * NG;
            const float4 v =
                b < nb ? __ldcg(reinterpret_cast<const float4 *>(x + 32L * b) + sub) : make_float4(0.f, 0.f, 0.f, 0.f);
            e[i][0] = v.x, e[i][1] = v.y, e[i][2] = v.z, e[i][3] = v.w;
        }
        if (b0 == 0) after_loads();
        float a[XCH];
#pragma unroll
        for (int i = 0; i < XCH; ++i)
            a[i] = fmaxf(fmaxf(fabsf(e[i][0]), fabsf(e[i][1])), fmaxf(fabsf(e[i][2]), fabsf(e[i][3])));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
#pragma unroll
            for (int i = 0; i < XCH; ++i) a[i] = fmaxf(a[i], __shfl_xor_sync(0xffffffffu, a[i], o));
        float d[XCH];
        int q[XCH][4];
        uint32_t need = 0;  // bit 4 i + k: element k of block i takes the rounded division
#pragma unroll
        for (int i = 0; i < XCH; ++i) {
            d[i] = __fdiv_rn(a[i], 127.0f);
            const float inv = __frcp_rn(d[i]);
            const bool div_only = d[i] < 1.17549435e-38f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // r: t rounded to the nearest integer (ties to even); where t is not within
                // 2^-14 of a half-integer that is also round(t) (ties away from zero)
                const float t = e[i][k] * inv;
                const int r = __float2int_rn(t);
                if (d[i] != 0.0f && (div_only || fabsf(t - (float)r) > 0.5f - 6.103515625e-05f))
                    need |= 1u << (4 * i + k);
                q[i][k] = d[i] != 0.0f && !div_only ? r : 0;
            }
        }
        if (__any_sync(0xffffffffu, need != 0)) {
#pragma unroll
            for (int i = 0; i < XCH; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if ((need >> (4 * i + k)) & 1u) q[i][k] = (int)roundf(__fdiv_rn(e[i][k], d[i]));
        }
        int sum[XCH], half[XCH];
#pragma unroll
        for (int i = 0; i < XCH; ++i) {
            sum[i] = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                q[i][k] = q[i][k] > 127 ? 127 : (q[i][k] < -127 ? -127 : q[i][k]);
                sum[i] += q[i][k];
            }
            half[i] = sub < 4 ? sum[i] : 0;  // elements 0..15 of the block
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
#pragma unroll
            for (int i = 0; i < XCH; ++i) {
                sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], o);
                half[i] += __shfl_xor_sync(0xffffffffu, half[i], o);
            }
#pragma unroll
        for (int i = 0; i < XCH; ++i) {
            const int b = b0 + grp + i * NG;
            if (b >= nb) continue;
            const uint32_t codes = (uint32_t)(q[i][0] & 0xff) | ((uint32_t)(q[i][1] & 0xff) << 8) |
                                   ((uint32_t)(q[i][2] & 0xff) << 16) | ((uint32_t)(q[i][3] & 0xff) << 24);
            const int u = b & (XGT - 1);
            uint8_t *t = xs + (size_t)(b / XGT) * STRIDE;
            reinterpret_cast<uint32_t *>(t + 32 * u)[sub] = codes;
            if (sub == 0) {
                reinterpret_cast<float *>(t + 32 * XGT)[u] = d[i];
                reinterpret_cast<int32_t *>(t + 36 * XGT)[u] = sum[i];
                reinterpret_cast<uint32_t *>(t + 40 * XGT)[u] =
                    ((uint32_t)half[i] & 0xffffu) | ((uint32_t)(sum[i] - half[i]) << 16);
                reinterpret_cast<float *>(t + 44 * XGT)[u] = d[i] * (float)sum[i];
            }
        }
    }
    // the repeated tiles: tile tpr + j is a copy of tile j mod tpr
    __syncthreads();
    repeat_tiles<STRIDE>(xs, tpr, xrep, tid, NTH);
}

// Tasks whose bytes make a multiple of 16: a warp's task range starts at a multiple of this
// many tasks, so that every stage (a whole number of such groups, or the rest of a range
// that ends on one) is a single 16-byte-aligned bulk copy of a 16-byte multiple.  1 for task
// sizes that are multiples of 16; 8 for Q6_K and Q3_K superblocks (210, 110 bytes).
__host__ __device__ constexpr int task_align_unit(int task_bytes) {
    return task_bytes % 16 == 0 ? 1 : task_bytes % 8 == 0 ? 2 : task_bytes % 4 == 0 ? 4 : task_bytes % 2 == 0 ? 8 : 16;
}
// The same for rows of rb bytes: CTA row ranges start at multiples of this many rows (2 for
// Q6_K rows of 5120 or 17408 elements, 4200 and 14280 bytes).
__host__ __device__ constexpr int row_align_unit(uint32_t rb) { return task_align_unit((int)(rb & 15u)); }

// shared memory: ring (S slots), activation tiles, partial sums, S + 1 mbarriers
__host__ __device__ constexpr uint32_t engine1_smem(int S, uint32_t slot_bytes, uint32_t x_bytes, int part_floats) {
    return (uint32_t)S * slot_bytes + x_bytes + 4u * (uint32_t)part_floats + 8u * (uint32_t)(S + 1) + 16u;
}

template <int FMT, int T, int NCW>
__global__ void __launch_bounds__(NCW * 32, 1) engine1_kernel(const Gemv1Args a) {
    using F = FT<FMT, T>;
    using TL = Tile<F::XGT>;
    constexpr uint32_t TB = F::TASK_BYTES;
    constexpr int AU = task_align_unit((int)TB);
    static_assert((32 * TB) % 16 == 0, "stages are single aligned bulk copies");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int D = a.depth, S = NCW * D;
    const uint32_t ring = smem_addr(smem);
    const uint32_t xa = ring + (uint32_t)S * a.slot_bytes;
    float *part = reinterpret_cast<float *>(smem + (uint32_t)S * a.slot_bytes + a.x_bytes);
    // tasks of a multiple of 16 bytes: rows too (ra = 1)
    const int o0 = AU == 1 ? split_point(a.N, (int)blockIdx.x, (int)gridDim.x)
                           : a.ra * split_point(a.nra, (int)blockIdx.x, (int)gridDim.x);
    const int o1 = AU == 1 ? split_point(a.N, (int)blockIdx.x + 1, (int)gridDim.x)
                           : a.ra * split_point(a.nra, (int)blockIdx.x + 1, (int)gridDim.x);
    const int tpr = a.tpr;
    const int ntask = (o1 - o0) * tpr;
    const uint32_t bars = ring + (uint32_t)S * a.slot_bytes + a.x_bytes + 4u * (uint32_t)ntask;
    const uint32_t bars8 = (bars + 7u) & ~7u;
    auto full_bar = [&](int s) { return bars8 + 8u * (uint32_t)s; };
    const uint32_t xbar = bars8 + 8u * (uint32_t)S;
    const uint8_t *base = a.W + (size_t)o0 * a.rb;

    griddep_launch_dependents();
    if (lane == 0) {
        for (int j = 0; j < D; ++j) mbar_init(full_bar(j * NCW + warp), 1);
        if (warp == 0) mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ntask is a multiple of AU (the CTA's rows make a multiple of 16 bytes)
    const int wa = AU * split_point(ntask / AU, warp, NCW), wb = AU * split_point(ntask / AU, warp + 1, NCW);
    const int nst = (wb - wa + 31) / 32;  // this warp's stages

    // stage j of this warp into its slot (lane 0; the slot must be free)
    auto issue = [&](int j) {
        if (lane == 0) {
            const int fa = wa + 32 * j, fb = min(wb, fa + 32);
            const uint32_t slot = (uint32_t)((j % D) * NCW + warp);
            const uint32_t bytes = (uint32_t)(fb - fa) * TB;
            bulk_g2s(ring + slot * a.slot_bytes, base + (size_t)fa * TB, bytes, full_bar((int)slot));
            mbar_arrive_expect_tx(full_bar((int)slot), bytes);
        }
    };
    // the first D stages; with x, right after the activation row's loads rather than before
    // them (a load queues behind the bulk copies this SM has in flight)
    const int jfirst = min(D, nst), jpre = a.x ? 0 : jfirst;
    for (int j = 0; j < jpre; ++j) issue(j);
    __syncthreads();
    if (a.x) {
        // the activation row, from the previous kernel: quantized here, by every thread
        griddep_wait();
        auto rest = [&] {
            for (int j = jpre; j < jfirst; ++j) issue(j);
        };
        if (ntask > 0) quant_row_tiles<F::XGT, NCW * 32>(a.x, a.K, smem + (xa - ring), tpr, a.xrep, tid, rest);
        __syncthreads();
    } else {
        if (warp == 0 && lane == 0) {
            griddep_wait();
            const uint32_t row_bytes = (uint32_t)tpr * TL::STRIDE;
            uint32_t tx = 0;
            if (ntask > 0) {
                bulk_g2s(xa, a.ximg, row_bytes, xbar);
                tx += row_bytes;
                // the row's first xrep tiles again after it
                for (int v = tpr; v < tpr + a.xrep; v += tpr) {
                    const uint32_t rb2 = (uint32_t)(min(tpr, tpr + a.xrep - v) * TL::STRIDE);
                    bulk_g2s(xa + (uint32_t)v * TL::STRIDE, a.ximg, rb2, xbar);
                    tx += rb2;
                }
            }
            mbar_arrive_expect_tx(xbar, tx);
        }
        mbar_wait(xbar, 0);
    }
    const FastDiv tpr_div = FastDiv::make((uint32_t)tpr);

    for (int j = 0; j < nst; ++j) {
        const int slot = (j % D) * NCW + warp;
        const int fa = wa + 32 * j, fb = min(wb, fa + 32);
        mbar_wait(full_bar(slot), (uint32_t)((j / D) & 1));
        const int f = fa + lane;
        const bool valid = f < fb;
        uint32_t w[F::WW];
        // a task starts 2-byte aligned at worst (Q6_K, Q3_K): the decoder realigns by aoff
        const uint32_t aoff = ((uint32_t)lane * TB) & 3u;
        if (valid) F::load(smem + (uint32_t)slot * a.slot_bytes + (uint32_t)lane * TB, w);
        __syncwarp();
        if (j + D < nst) {
            fence_proxy_async_smem();
            issue(j + D);
        }
        if (valid) {
            const int o = (int)tpr_div.div((uint32_t)f), tt = f - o * tpr;
            // with repeated tiles lane l reads virtual column (column of the stage's first
            // task) + l, past the row's end where the stage wraps
            const int xc = a.xrep ? fa - (int)tpr_div.div((uint32_t)fa) * tpr + lane : tt;
            AccSink<1> sink;
            sink.acc[0] = 0.0f;
            F::compute(w, aoff, tt % F::TPB, XT{smem + (xa - ring) + (uint32_t)(xc * TL::STRIDE), 0u}, 1, sink);
            part[f] = sink.acc[0];
        }
    }
    // every stage was consumed; copies still in flight after a wait gave up land first
    if (lane == 0) {
        for (int d = 0; d < D && d < nst; ++d)
            mbar_drain(full_bar(d * NCW + warp), (uint32_t)(((d + D * ((nst - 1 - d) / D)) / D) & 1), DRAIN_NS);
        if (warp == 0 && !a.x) mbar_drain(xbar, 0, DRAIN_NS);
    }
    __syncthreads();
    for (int r = tid; r < o1 - o0; r += NCW * 32) {
        const float *p = part + (size_t)r * tpr;
        float s = 0.0f;
        for (int t = 0; t < tpr; ++t) s += p[t];
        a.y[o0 + r] = s;
    }
}

}  // namespace qg

namespace qg {

// The FFN sublayer's gate and up projections at one token with SwiGLU and the
// requantization of h in the epilogue ("为什么专家缓存救不了稠密模型", "原位量化计算与单流
// 融合的实际收益": the sublayer on one stream).  A CTA owns whole units of 32 positions j of
// the intermediate (rows 32 u .. 32 u + 31 of Wg and of Wu): its gate rows and its up rows
// are two contiguous byte ranges, consumed as in engine1_kernel (a stage that crosses from
// the gate range to the up range is two bulk copies).  After the last stage the CTA adds
// each row's partial sums in task order (g and u), forms h = silu(g) u, quantizes every
// unit of h as one activation block and writes it into the down projection's tile image,
// so the down GEMV needs no preparation kernel; g, u and h also go to the workspace.
struct FfnGateUp1Args {
    const uint8_t *Wg, *Wu;  // I rows of rb bytes each
    const uint8_t *ximg;     // activation tile image of x: tpr tiles
    const float *x;          // or (non-null): the fp32 row of K elements, quantized by every CTA
    int K;
    float *g_out, *u_out, *h_out;
    uint8_t *himg;           // the down projection's tile image (one row)
    int I, tpr, depth, xrep, himg_tpr, himg_xgt_log2;
    uint32_t rb, slot_bytes, x_bytes;
};

// partial sums of a CTA with nu units: 2 * 32 * nu rows of tpr tasks, then 2 * 32 * nu row sums
__host__ __device__ constexpr int ffn1_part_floats(int nu, int tpr) { return 64 * nu * tpr + 64 * nu; }

template <int FMT, int T, int NCW>
__global__ void __launch_bounds__(NCW * 32, 1) ffn_gateup1_kernel(const FfnGateUp1Args a) {
    using F = FT<FMT, T>;
    using TL = Tile<F::XGT>;
    constexpr uint32_t TB = F::TASK_BYTES;
    constexpr int AU = task_align_unit((int)TB);
    static_assert((32 * TB) % 16 == 0, "stages are aligned bulk copies");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int D = a.depth, S = NCW * D;
    const uint32_t ring = smem_addr(smem);
    const uint32_t xa = ring + (uint32_t)S * a.slot_bytes;
    float *part = reinterpret_cast<float *>(smem + (uint32_t)S * a.slot_bytes + a.x_bytes);
    const int U = a.I / 32;
    const int u0 = split_point(U, (int)blockIdx.x, (int)gridDim.x);
    const int u1 = split_point(U, (int)blockIdx.x + 1, (int)gridDim.x);
    const int nu = u1 - u0, nr = 32 * nu, tpr = a.tpr;
    const int G = nr * tpr, ntask = 2 * G;  // gate tasks [0, G), up tasks [G, 2G)
    float *rsum = part + ntask;             // row sums: gate rows, then up rows
    const uint32_t bars = smem_addr(part + ffn1_part_floats(nu, tpr));
    const uint32_t bars8 = (bars + 7u) & ~7u;
    auto full_bar = [&](int s) { return bars8 + 8u * (uint32_t)s; };
    const uint32_t xbar = bars8 + 8u * (uint32_t)S;
    const uint8_t *gbase = a.Wg + (size_t)(32 * u0) * a.rb, *ubase = a.Wu + (size_t)(32 * u0) * a.rb;

    griddep_launch_dependents();
    if (lane == 0) {
        for (int j = 0; j < D; ++j) mbar_init(full_bar(j * NCW + warp), 1);
        if (warp == 0) mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // G (whole rows) is a multiple of AU: so are the warp ranges and the gate/up boundary
    const int wa = AU * split_point(ntask / AU, warp, NCW), wb = AU * split_point(ntask / AU, warp + 1, NCW);
    const int nst = (wb - wa + 31) / 32;

    auto issue = [&](int j) {
        if (lane == 0) {
            const int fa = wa + 32 * j, fb = min(wb, fa + 32);
            const uint32_t slot = (uint32_t)((j % D) * NCW + warp);
            const uint32_t dst = ring + slot * a.slot_bytes;
            const int g1 = min(fb, G);  // gate tasks [fa, g1), up tasks [max(fa, G), fb)
            uint32_t bytes = 0;
            if (fa < g1) {
                bulk_g2s(dst, gbase + (size_t)fa * TB, (uint32_t)(g1 - fa) * TB, full_bar((int)slot));
                bytes += (uint32_t)(g1 - fa) * TB;
            }
            const int ua = max(fa, G);
            if (ua < fb) {
                bulk_g2s(dst + bytes, ubase + (size_t)(ua - G) * TB, (uint32_t)(fb - ua) * TB, full_bar((int)slot));
                bytes += (uint32_t)(fb - ua) * TB;
            }
            mbar_arrive_expect_tx(full_bar((int)slot), bytes);
        }
    };
    // as in engine1_kernel: with x, the first stages go out right after the row's loads
    const int jfirst = min(D, nst), jpre = a.x ? 0 : jfirst;
    for (int j = 0; j < jpre; ++j) issue(j);
    __syncthreads();
    if (a.x) {
        griddep_wait();
        auto rest = [&] {
            for (int j = jpre; j < jfirst; ++j) issue(j);
        };
        if (ntask > 0) quant_row_tiles<F::XGT, NCW * 32>(a.x, a.K, smem + (xa - ring), tpr, a.xrep, tid, rest);
        __syncthreads();
    } else {
        if (warp == 0 && lane == 0) {
            griddep_wait();
            const uint32_t row_bytes = (uint32_t)tpr * TL::STRIDE;
            uint32_t tx = 0;
            if (ntask > 0) {
                bulk_g2s(xa, a.ximg, row_bytes, xbar);
                tx += row_bytes;
                for (int v = tpr; v < tpr + a.xrep; v += tpr) {
                    const uint32_t rb2 = (uint32_t)(min(tpr, tpr + a.xrep - v) * TL::STRIDE);
                    bulk_g2s(xa + (uint32_t)v * TL::STRIDE, a.ximg, rb2, xbar);
                    tx += rb2;
                }
            }
            mbar_arrive_expect_tx(xbar, tx);
        }
        mbar_wait(xbar, 0);
    }
    const FastDiv tpr_div = FastDiv::make((uint32_t)tpr);

    for (int j = 0; j < nst; ++j) {
        const int slot = (j % D) * NCW + warp;
        const int fa = wa + 32 * j, fb = min(wb, fa + 32);
        mbar_wait(full_bar(slot), (uint32_t)((j / D) & 1));
        const int f = fa + lane;
        const bool valid = f < fb;
        uint32_t w[F::WW];
        const uint32_t aoff = ((uint32_t)lane * TB) & 3u;
        if (valid) F::load(smem + (uint32_t)slot * a.slot_bytes + (uint32_t)lane * TB, w);
        __syncwarp();
        if (j + D < nst) {
            fence_proxy_async_smem();
            issue(j + D);
        }
        if (valid) {
            // G is a multiple of tpr: a task's column is its index modulo tpr in both ranges
            const int o = (int)tpr_div.div((uint32_t)f), tt = f - o * tpr;
            const int xc = a.xrep ? fa - (int)tpr_div.div((uint32_t)fa) * tpr + lane : tt;
            AccSink<1> sink;
            sink.acc[0] = 0.0f;
            F::compute(w, aoff, tt % F::TPB, XT{smem + (xa - ring) + (uint32_t)(xc * TL::STRIDE), 0u}, 1, sink);
            part[f] = sink.acc[0];
        }
    }
    if (lane == 0) {
        for (int d = 0; d < D && d < nst; ++d)
            mbar_drain(full_bar(d * NCW + warp), (uint32_t)(((d + D * ((nst - 1 - d) / D)) / D) & 1), DRAIN_NS);
        if (warp == 0 && !a.x) mbar_drain(xbar, 0, DRAIN_NS);
    }
    __syncthreads();
    // row sums in task order: g of the CTA's gate rows, then u of its up rows
    for (int r = tid; r < 2 * nr; r += NCW * 32) {
        const float *p = part + (size_t)r * tpr;
        float s = 0.0f;
        for (int t = 0; t < tpr; ++t) s += p[t];
        rsum[r] = s;
    }
    __syncthreads();
    // per unit: h = silu(g) u, quantized as one activation block into the down tile image
    for (int u = warp; u < nu; u += NCW) {
        const int j = 32 * (u0 + u) + lane;
        const float g = rsum[32 * u + lane], uu = rsum[nr + 32 * u + lane];
        const float h = silu_mul(g, uu);
        a.g_out[j] = g;
        a.u_out[j] = uu;
        a.h_out[j] = h;
        int q, s;
        float d;
        quant_block_warp(h, q, d, s);
        put_block(a.himg, 0, a.himg_tpr, u0 + u, a.himg_xgt_log2, lane, q, d, s);
    }
}

}  // namespace qg
