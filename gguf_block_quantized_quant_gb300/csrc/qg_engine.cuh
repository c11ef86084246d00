// qg_engine.cuh -- the weight-streaming engine behind every GEMV-shaped kernel of libqg.
//
// Decode GEMV is bound by HBM bandwidth: every weight byte is read once and used for
// M <= 16 tokens.  The engine keeps enough bytes in flight per SM and spends as few
// instructions per weight byte as it can.
//
// Work model.  A job is a sequence of OUTPUT ROWS, each the dot product of one weight-matrix
// row (tpr tasks, see qg_formats.cuh) with an activation row.  Rows come in groups of grp
// consecutive rows that are adjacent in memory (a whole matrix for a plain GEMV).
//
//  * one CTA per SM (persistent) with NCW warps; the CTA owns a contiguous range of output
//    rows (and, for split-K, a slice of every row);
//  * the CTA's tasks are split into NCW contiguous ranges, one per warp; a warp consumes
//    its range in stages of tps tasks, lane l of step s taking task 32 s + l;
//  * every warp feeds itself: it owns D slots of the shared-memory ring (its j-th stage
//    lands in slot (j mod D) * NCW + w), issues its first D stages up front, and refills a
//    slot with stage j + D as soon as it has consumed stage j.  A stage is copied with 1-D
//    bulk copies (cp.async.bulk, the TMA engine), one per run of adjacent rows, issued by
//    up to NPIECE_MAX lanes in parallel; completion is counted in bytes on the slot's
//    mbarrier.  Pieces that start or end off a 16-byte boundary are widened to it, and
//    bytes past the end of a tensor that the widened copy may not read are loaded one by
//    one.  No warp ever waits for another warp's progress to get its data;
//  * activations arrive as a tile image written once per call by a preparation kernel;
//    warp 0 issues its first stages, then waits for that kernel (programmatic dependent
//    launch) and copies the image rows the CTA needs into shared memory.  The engine in
//    turn lets the next call's preparation launch early, so back-to-back calls overlap
//    one call's tail with the next call's weight streaming;
//  * a lane decodes its task in registers against the activation tiles; per step, a
//    segmented shuffle reduction (rows are contiguous runs of lanes) leaves each row's
//    sum at the row's first lane; a row that continues in the warp's next step is carried
//    in registers; complete rows are stored by the job; rows shared with the neighbouring
//    warp are combined after the last stage, in warp order, so every result is
//    deterministic; the job may finish with a CTA-wide epilogue (MoE weighted sums).
#pragma once

#include "qg_formats.cuh"

namespace qg {

constexpr int NPIECE_MAX = 8;      // weight pieces per stage
// Prologue scratch: the MoE launches' routed expert ids (up to SCRATCH_W of them), and in
// the down launch their routing weights (float bits) from SCRATCH_W on.
constexpr int SCRATCH_W = 256;
constexpr int SCRATCH_INTS = 2 * SCRATCH_W;
constexpr int BND_FLOATS = 1 + 16; // boundary entry: row, then one sum per token

// Unsigned division by a run-time constant (n < 2^31, d < 2^31): 32-bit reciprocal
// estimate m = ceil(2^32 / d) (any m in [2^32 / d, 2^32 / d + 2) gives a quotient that is
// exact or one too large for n < 2^31), corrected once.  m comes from a 32-bit division:
// (2^32 - 1) / d + 1 equals ceil(2^32 / d) for every d > 1.
struct FastDiv {
    uint32_t d, m;
    __host__ __device__ static FastDiv make(uint32_t dv) {
        FastDiv f;
        f.d = dv;
        f.m = dv <= 1 ? 0u : 0xffffffffu / dv + 1u;
        return f;
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        if (d <= 1) return n;
        uint32_t q = __umulhi(n, m);
        if (q * d > n) --q;
        return q;
    }
};

// floor(n * i / parts) for 0 <= i <= parts (the start of part i when n items are split into
// parts nearly equal parts): 32-bit arithmetic whenever n * parts < 2^32, which holds for
// every planned shape (a 64-bit division is a long call on the GPU, and every thread of a
// CTA computes its range before its first copy).
__device__ __forceinline__ int split_point(long n, int i, int parts) {
    if ((unsigned long long)n * (unsigned long long)parts < (1ull << 32))
        return (int)((uint32_t)n * (uint32_t)i / (uint32_t)parts);
    return (int)(n * i / parts);
}

// Shared memory of the engine besides the ring, the activation tiles and the job area:
// boundary sums (2 per warp), prologue scratch, S + 1 mbarriers, piece headers (per slot:
// NPIECE_MAX piece addresses and the end of the tasks the pieces cover).
__host__ __device__ constexpr uint32_t engine_fixed_smem(int S, int ncw) {
    return (uint32_t)(ncw * 2 * BND_FLOATS * 4) + 4u * SCRATCH_INTS + 8u * (uint32_t)S + 8u +
           4u * (NPIECE_MAX + 1) * (uint32_t)S + 16u;
}

// Byte offset of task tt within a row (tasks are whole blocks, or half a superblock).
template <class F>
__host__ __device__ __forceinline__ uint32_t task_off(int tt) {
    return (uint32_t)((tt / F::TPB) * F::BPT * F::BS);
}

// GEMV sink: per-token fp32 accumulators of one lane.
template <int NT>
struct AccSink {
    static constexpr int MT = NT;
    static constexpr bool DOTS = false;
    float acc[NT];
    __device__ __forceinline__ void add(int m, float v) { acc[m] += v; }
};

// Orders this thread's earlier generic-proxy accesses of shared memory before its later
// async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// NCW: warps of the CTA (engine_ncw(), or 12 for large one-token launches, see plan_ncw).
template <int FMT, int T, int MT, int NCW, class Job>
__global__ void __launch_bounds__(NCW * 32, 1) engine_kernel(const Job job) {
    using F = FT<FMT, T>;
    using TL = Tile<F::XGT>;
    constexpr int NCONS = NCW * 32;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int D = job.depth, S = NCW * D;
    const uint32_t slot_stride = job.slot_bytes + STAGE_SLACK;

    const uint32_t ring = smem_addr(smem);
    const uint32_t xa = ring + (uint32_t)S * slot_stride;              // activation tiles
    const uint32_t ja = xa + job.x_bytes;                              // job area
    const uint32_t bnd = ja + job.j_bytes;                             // boundary sums
    const uint32_t scr = bnd + (uint32_t)(NCW * 2 * BND_FLOATS * 4);   // prologue scratch
    const uint32_t bars = scr + 4u * SCRATCH_INTS;
    const uint32_t xbar = bars + 8u * (uint32_t)S;
    const uint32_t hdrs = xbar + 8u;
    auto full_bar = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto hdr = [&](int s, int p) { return hdrs + 4u * (uint32_t)(s * (NPIECE_MAX + 1) + p); };
    const uint32_t tok_stride = (uint32_t)((job.tpr_x + job.xrep) * TL::STRIDE);
    float *bsum = reinterpret_cast<float *>(smem + (bnd - ring));  // [NCW][2][BND_FLOATS]
    int *scratch = reinterpret_cast<int *>(smem + (scr - ring));
    float *jarea = reinterpret_cast<float *>(smem + (ja - ring));

    // the next kernel in the stream (the next call's activation preparation, launched as a
    // programmatic dependent) may start now: it waits for this grid to finish before it
    // touches any data, and its own dependent engine takes each SM this CTA leaves
    griddep_launch_dependents();
    // every warp initialises the barriers of its own ring slots (so that it can issue its
    // first copies before the CTA-wide barrier), warp 0 also the activation barrier
    if (lane == 0) {
        for (int j = 0; j < D; ++j) mbar_init(full_bar(j * NCW + warp), 1);
        if (warp == 0) mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // this CTA's tasks and this warp's range (whole blocks)
    const typename Job::Ctx cx = job.ctx();
    int o0, o1, tpr, grp;
    job.cta(cx, o0, o1, tpr, grp);
    const int ntask = (o1 - o0) * tpr;
    const FastDiv tpr_div = FastDiv::make((uint32_t)tpr), grp_div = FastDiv::make((uint32_t)grp);
    const int units = ntask / F::TPB;
    auto wstart = [&](int w) { return (int)((long)units * w / NCW) * F::TPB; };
    const int maxlen = (units + NCW - 1) / NCW * F::TPB;
    const int nchunk = (maxlen + job.tps - 1) / job.tps;
    const int a = wstart(warp), b = wstart(warp + 1);

    // Copies stage j of this warp into its slot; all 32 lanes take part (lane p < NPIECE_MAX
    // copies the stage's p-th run of adjacent rows).  The slot must be free.
    auto issue = [&](int j) {
        const int slot = (j % D) * NCW + warp;
        const int fa = a + j * job.tps, fb = min(b, fa + job.tps);
        const uint32_t sbase = ring + (uint32_t)slot * slot_stride;
        const uint32_t fbar = full_bar(slot);
        int ps = fa, pe = fa;  // this lane's piece [ps, pe)
        int covered = fb;
        if (fa < fb) {
            if (grp == 0) {
                if (lane == 0) pe = fb;
            } else {
                const int oa = (int)tpr_div.div((uint32_t)fa);
                const int ga = (int)grp_div.div((uint32_t)(o0 + oa));
                const long g0 = (long)(ga + lane) * grp - o0;  // first CTA-relative row of group ga + lane
                const long lo = g0 * tpr, hi = (g0 + grp) * tpr;
                if (lane < NPIECE_MAX) {
                    ps = (int)max((long)fa, lo);
                    pe = (int)min((long)fb, hi);
                }
                const long cend = ((long)(ga + NPIECE_MAX) * grp - o0) * tpr;  // end of the last piece's group
                if (cend < fb) {
                    // the stage needs more pieces than the table holds (a planning error):
                    // the rest of it is skipped and the host sees DEVERR_PLAN
                    covered = (int)cend;
                    if (lane == 0) atomicOr(&g_qg_dev_err, DEVERR_PLAN);
                }
            }
        }
        const bool valid = ps < pe;
        uintptr_t s0 = 0, a0 = 0, e = 0, a1 = 0, a1c = 0;
        if (valid) {
            const int o = (int)tpr_div.div((uint32_t)ps), tt = ps - o * tpr;
            const uint8_t *lim;
            const uint8_t *src = job.seg_src(cx, o0 + o, tt, lim, scratch);
            s0 = (uintptr_t)src;
            a0 = s0 & ~(uintptr_t)15;
            e = s0 + task_off<F>(pe - ps);
            a1 = (e + 15) & ~(uintptr_t)15;
            const uintptr_t lim16 = (uintptr_t)lim & ~(uintptr_t)15;
            a1c = a1 <= lim16 ? a1 : lim16;
            if (a1c < a0) a1c = a0;
        }
        // slot offsets: exclusive prefix sum of the widened piece sizes over the lanes
        const uint32_t wsz = (uint32_t)(a1 - a0);
        uint32_t incl = wsz;
#pragma unroll
        for (int d = 1; d < NPIECE_MAX; d <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        const uint32_t off = incl - wsz;
        const uint32_t nb = (uint32_t)(a1c - a0);
        if (valid) {
            for (uintptr_t q = a1c; q < e; ++q)
                sts8(sbase + off + (uint32_t)(q - a0), *reinterpret_cast<const uint8_t *>(q));
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(hdr(slot, lane)), "r"(sbase + off + (uint32_t)(s0 & 15))
                         : "memory");
            if (nb) bulk_g2s(sbase + off, reinterpret_cast<const void *>(a0), nb, fbar);
        }
        const uint32_t tx = __reduce_add_sync(0xffffffffu, nb);
        if (lane == 0)
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(hdr(slot, NPIECE_MAX)), "r"(covered) : "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(fbar, tx);
    };

    // the first D stages: the slots are free.  A job with a prologue (whose copies depend
    // on it) issues them after the CTA-wide set-up, any other job before it.
    const int jfirst = min(D, nchunk);
    if constexpr (!Job::HAS_PROLOGUE)
        for (int j = 0; j < jfirst; ++j) issue(j);
    if (tid < NCW * 2) bsum[tid * BND_FLOATS] = __int_as_float(-1);
    job.init(jarea, tid);
    if constexpr (Job::HAS_PROLOGUE) {
        __syncthreads();
        job.prologue(warp, NCW, lane, scratch);
    }
    __syncthreads();
    // the activation tiles (their own copies, after the previous kernel has finished); a job
    // with a prologue issues them before its weight stages, which the prologue also gated
    if (warp == 0) {
        if (lane == 0) {
            griddep_wait();
            const int rows = ntask > 0 ? job.xrows() : 0;
            uint32_t tx = 0;
            for (int r = 0; r < rows; ++r) {
                const uint32_t bytes = job.xrow_bytes(cx, r);
                if (bytes) bulk_g2s(xa + (uint32_t)r * tok_stride, job.xrow_src(cx, r), bytes, xbar);
                tx += bytes;
                // the row's first job.xrep tiles again after it (the row holds tpr tiles)
                for (int v = tpr; v < tpr + job.xrep; v += tpr) {
                    const uint32_t rb2 = (uint32_t)(min(tpr, tpr + job.xrep - v) * TL::STRIDE);
                    bulk_g2s(xa + (uint32_t)r * tok_stride + (uint32_t)(v * TL::STRIDE), job.xrow_src(cx, r), rb2,
                             xbar);
                    tx += rb2;
                }
            }
            mbar_arrive_expect_tx(xbar, tx);
        }
        __syncwarp();
    }
    if constexpr (Job::HAS_PROLOGUE)
        for (int j = 0; j < jfirst; ++j) issue(j);

    // ---------------------------------------------------------------------- consume
    const int ra = (int)tpr_div.div((uint32_t)a);
    const bool a_mid = a < b && a != ra * tpr;
    const int ntok = job.ntok;
    mbar_wait(xbar, 0);

    float carry[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) carry[m] = 0.0f;
    int carry_o = -1;  // CTA-relative output row whose partial sum is in carry

    for (int j = 0; j < nchunk; ++j) {
        const int slot = (j % D) * NCW + warp;
        const int fa = a + j * job.tps;  // a stage is at most 32 tasks: one per lane
        mbar_wait(full_bar(slot), (uint32_t)((j / D) & 1));
        const int fb = min(min(b, fa + job.tps), (int)lds32(hdr(slot, NPIECE_MAX)));
        const int f = fa + lane;
        const bool valid = f < fb;
        int o = 0x7fffffff, tt = 0;
        uint32_t w[F::WW];
        uint32_t aoff = 0;
        SAddr xbase = smem;
        if (valid) {
            o = (int)tpr_div.div((uint32_t)f);
            tt = f - o * tpr;
            int piece = 0, fp = fa;
            if (grp) {
                const int ga = (int)grp_div.div((uint32_t)(o0 + (int)tpr_div.div((uint32_t)fa)));
                const int g = (int)grp_div.div((uint32_t)(o0 + o));
                piece = g - ga;
                if (piece) fp = (g * grp - o0) * tpr;
            }
            const SAddr addr = smem + (lds32(hdr(slot, piece)) - ring) + task_off<F>(f - fp);
            F::load(addr, w);
            aoff = (uint32_t)((uintptr_t)addr & 3u);
            // with repeated tiles a lane reads virtual column (column of the stage's first
            // task) + lane, past the row's end where the stage wraps
            const int xc = job.xrep ? fa - (int)tpr_div.div((uint32_t)fa) * tpr + lane : tt;
            xbase = smem + (xa - ring) + job.xrow(cx, o0 + o, grp_div) * tok_stride + (uint32_t)(xc * TL::STRIDE);
        }
        // the stage is in registers: refill the slot with stage j + D while decoding
        __syncwarp();
        if (j + D < nchunk) {
            fence_proxy_async_smem();
            issue(j + D);
        }
        if (fa < fb) {
            const int f0 = fa;
            AccSink<MT> sink;
#pragma unroll
            for (int m = 0; m < MT; ++m) sink.acc[m] = 0.0f;
            if (valid) F::compute(w, aoff, tt % F::TPB, XT{xbase, tok_stride}, ntok, sink);
            // segmented reduction: rows are contiguous runs of lanes
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o2 = __shfl_down_sync(0xffffffffu, o, d);
                const bool take = lane + d < 32 && o2 == o;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float v = __shfl_down_sync(0xffffffffu, sink.acc[m], d);
                    if (take) sink.acc[m] += v;
                }
            }
            const int oprev = __shfl_up_sync(0xffffffffu, o, 1);
            const bool head = valid && (lane == 0 || oprev != o);
            if (head && o == carry_o) {
#pragma unroll
                for (int m = 0; m < MT; ++m) sink.acc[m] += carry[m];
            }
            // the step's last row continues if it has tasks after this step
            const int flast = min(fb, f0 + 32) - 1;
            const int olast = __shfl_sync(0xffffffffu, o, flast - f0);
            const bool cont = (olast + 1) * tpr > flast + 1;
            if (head && !(o == olast && cont)) {
                if (a_mid && o == ra) {
                    float *e = bsum + (warp * 2) * BND_FLOATS;  // shared with the previous warp
                    e[0] = __int_as_float(o);
#pragma unroll
                    for (int m = 0; m < MT; ++m) e[1 + m] = sink.acc[m];
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < ntok) job.store(cx, o0 + o, m, sink.acc[m], jarea);
                }
            }
            // the continuing row's head broadcasts its sums as the next carry
            const int hl = __reduce_min_sync(0xffffffffu, (valid && o == olast) ? lane : 31);
#pragma unroll
            for (int m = 0; m < MT; ++m) carry[m] = __shfl_sync(0xffffffffu, sink.acc[m], hl);
            carry_o = cont ? olast : -1;
        }
    }
    // every stage was consumed on the normal path; after a wait gave up, this warp's bulk
    // copies still in flight land (bounded) before the CTA can exit
    if (lane == 0) {
        for (int d = 0; d < D && d < nchunk; ++d)
            mbar_drain(full_bar(d * NCW + warp), (uint32_t)(((d + D * ((nchunk - 1 - d) / D)) / D) & 1), DRAIN_NS);
        if (warp == 0) mbar_drain(xbar, 0, DRAIN_NS);
    }
    // a range that ended inside a row: its sum is shared with the next warp
    if (carry_o >= 0 && lane == 0) {
        float *e = bsum + (warp * 2 + ((a_mid && carry_o == ra) ? 0 : 1)) * BND_FLOATS;
        e[0] = __int_as_float(carry_o);
#pragma unroll
        for (int m = 0; m < MT; ++m) e[1 + m] = carry[m];
    }
    consumer_sync<NCONS>();
    // rows shared by consecutive warps: their sums added in warp order.  Lane l of warp 0
    // holds boundary entry l (warp l / 2, side l % 2); the entries of one row are the lanes
    // that match its index (they are consecutive among the used entries, as the warps' rows
    // ascend), and the first of them adds them up in lane order and stores the sums.
    static_assert(2 * NCW <= 32, "one lane per boundary entry");
    if (warp == 0) {
        const int r = lane < 2 * NCW ? __float_as_int(bsum[lane * BND_FLOATS]) : -1;
        const uint32_t same = __match_any_sync(0xffffffffu, r);
        if (r >= 0 && lane == __ffs(same) - 1) {
            for (int m = 0; m < ntok; ++m) {
                float acc = 0.0f;
                for (uint32_t k = same; k; k &= k - 1) acc += bsum[(__ffs(k) - 1) * BND_FLOATS + 1 + m];
                job.store(cx, o0 + r, m, acc, jarea);
            }
        }
    }
    if (Job::HAS_FINISH) {
        consumer_sync<NCONS>();
        job.finish(cx, jarea, tid, NCONS, scratch);
    }
}


// ===================================================================================
// Row-pair engine (plain GEMV with whole rows per CTA).  A task is the same column block
// of two adjacent rows (one superblock, or 4 or 8 32-element blocks, of each), so every
// activation-tile load of a lane serves both rows: half the tile traffic of one-row tasks
// of the same size (and Q4_K / Q4_0 tasks 144 bytes apart, an odd number of 16-byte
// chunks, load without bank conflicts).  The CTA owns row pairs [p0, p1); tasks are
// ordered pair by pair, column by column.  A stage's bytes are at most three runs of the
// row-major matrix: the first pair's first row from the stage's first column, everything
// from that pair's second row (same column) through the last pair's first row, and the
// last pair's second row up to the stage's last column.  Ring, barriers, refill, carries
// and the combine of pairs shared by two warps work as in engine_kernel, with two sums
// per token.
constexpr int PAIR_BND = 1 + 2 * 16;  // boundary entry: pair, then row-0 and row-1 sums
constexpr int PAIR_RUNS = 3;        // runs of a stage over whole rows
constexpr int PAIR_RUNS_SPLIT = 8;  // over K-slices: one run per row of up to 4 pairs
constexpr int PAIR_SPLIT_MIN_TPR = 11;  // slice tasks that keep a 32-task stage within 4 pairs
__host__ __device__ constexpr uint32_t pair_fixed_smem(int S, int ncw) {
    return (uint32_t)(ncw * 2 * PAIR_BND * 4) + 8u * (uint32_t)S + 8u + 4u * PAIR_RUNS_SPLIT * (uint32_t)S + 16u;
}

template <int NT>
struct PairSink {
    static constexpr int MT = NT;
    float acc[2][NT];
    __device__ __forceinline__ void add(int r, int m, float v) { acc[r][m] += v; }
};

template <int FMT, int T, int MT, int NCW, class Job>
__global__ void __launch_bounds__(NCW * 32, 1) engine_pair_kernel(const Job job) {
    using F = FT<FMT, T>;
    using TL = Tile<F::XGT>;
    constexpr int NCONS = NCW * 32;
    constexpr uint32_t TB = F::TASK_BYTES;  // one row's part of a task
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int D = job.depth, S = NCW * D;
    const uint32_t slot_stride = job.slot_bytes + STAGE_SLACK;

    const uint32_t ring = smem_addr(smem);
    const uint32_t xa = ring + (uint32_t)S * slot_stride;             // activation tiles
    const uint32_t bnd = xa + job.x_bytes;                            // boundary sums
    const uint32_t bars = bnd + (uint32_t)(NCW * 2 * PAIR_BND * 4);
    const uint32_t xbar = bars + 8u * (uint32_t)S;
    const uint32_t hdrs = xbar + 8u;
    auto full_bar = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto hdr = [&](int s, int k) { return hdrs + 4u * (uint32_t)(s * PAIR_RUNS_SPLIT + k); };
    const uint32_t tok_stride = (uint32_t)(job.tpr_x * TL::STRIDE);
    float *bsum = reinterpret_cast<float *>(smem + (bnd - ring));  // [NCW][2][PAIR_BND]

    griddep_launch_dependents();
    if (lane == 0) {
        for (int j = 0; j < D; ++j) mbar_init(full_bar(j * NCW + warp), 1);
        if (warp == 0) mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // CTA = (group of row pairs, K-slice): with KS > 1 the CTA takes tasks [t0, t0 + tpr)
    // of every row of its pairs and writes partial sums to slice ks of job.out
    const int N = job.N, KS = job.KS;
    const bool split = KS > 1;
    const int grp = (int)blockIdx.x / KS, ks = (int)blockIdx.x - grp * KS, ngroups = (int)gridDim.x / KS;
    const int t0 = split_point(job.gpr, ks, KS) * F::TPB;
    const int tpr = split_point(job.gpr, ks + 1, KS) * F::TPB - t0;
    float *const out = job.out + (long)ks * job.slice_stride;
    const int P = (N + 1) >> 1;
    const int p0 = split_point(P, grp, ngroups);
    const int p1 = split_point(P, grp + 1, ngroups);
    const int ntask = (p1 - p0) * tpr;
    const FastDiv tpr_div = FastDiv::make((uint32_t)tpr);
    const int a = (int)((long)ntask * warp / NCW), b = (int)((long)ntask * (warp + 1) / NCW);
    const int maxlen = (ntask + NCW - 1) / NCW;
    const int nchunk = (maxlen + job.tps - 1) / job.tps;

    // Copies stage j of this warp into its slot (which must be free).  Whole rows: lane
    // k < 3 copies run k (see above).  K-slices: lane k < 8 copies the slice part of row
    // k & 1 of the stage's (k >> 1)-th pair.
    auto issue = [&](int j) {
        const int slot = (j % D) * NCW + warp;
        const int fa = a + j * job.tps, fb = min(b, fa + job.tps);
        const uint32_t sbase = ring + (uint32_t)slot * slot_stride;
        const uint32_t fbar = full_bar(slot);
        bool valid = false;
        uintptr_t s0 = 0, a0 = 0, e = 0, a1c = 0;
        if (fa < fb && lane < (split ? PAIR_RUNS_SPLIT : PAIR_RUNS)) {
            const int pa = (int)tpr_div.div((uint32_t)fa), ca = fa - pa * tpr;
            const int pb = (int)tpr_div.div((uint32_t)(fb - 1)), cb = fb - 1 - pb * tpr;
            const int ra = 2 * (p0 + pa), rz = 2 * (p0 + pb);
            int row = 0, col = 0, n = 0;
            if (split) {
                const int pp = pa + (lane >> 1);
                if (pp <= pb) {
                    row = 2 * (p0 + pp) + (lane & 1);
                    col = pp == pa ? ca : 0;
                    n = (pp == pb ? cb + 1 : tpr) - col;
                }
                // a stage over more than 4 pairs (a planning error) is skipped past them
                if (lane == 0 && pb - pa >= PAIR_RUNS_SPLIT / 2) atomicOr(&g_qg_dev_err, DEVERR_PLAN);
            } else if (lane == 0) {
                row = ra, col = ca, n = pa == pb ? cb - ca + 1 : tpr - ca;
            } else if (lane == 1) {
                row = ra + 1, col = ca;
                n = pa == pb ? cb - ca + 1 : (tpr - ca) + (rz - ra - 2) * tpr + cb + 1;
            } else if (pb > pa) {
                row = rz + 1, col = 0, n = cb + 1;
            }
            valid = n > 0 && row < N;
            if (valid) {
                s0 = (uintptr_t)(job.W + (size_t)row * job.rb + (size_t)(t0 + col) * TB);
                a0 = s0 & ~(uintptr_t)15;
                e = s0 + (uintptr_t)n * TB;
                const uintptr_t lim16 = (uintptr_t)job.Wend & ~(uintptr_t)15;
                a1c = (e + 15) & ~(uintptr_t)15;
                if (a1c > lim16) a1c = lim16 > a0 ? lim16 : a0;
            }
        }
        // slot offsets: exclusive prefix sum of the widened run sizes over lanes 0..2
        const uint32_t wsz = valid ? (uint32_t)(((e + 15) & ~(uintptr_t)15) - a0) : 0u;
        uint32_t incl = wsz;
#pragma unroll
        for (int d = 1; d < PAIR_RUNS_SPLIT; d <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        const uint32_t off = incl - wsz;
        const uint32_t nb = valid ? (uint32_t)(a1c - a0) : 0u;
        if (valid) {
            for (uintptr_t q = a1c; q < e; ++q)
                sts8(sbase + off + (uint32_t)(q - a0), *reinterpret_cast<const uint8_t *>(q));
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(hdr(slot, lane)), "r"(sbase + off + (uint32_t)(s0 & 15))
                         : "memory");
            if (nb) bulk_g2s(sbase + off, reinterpret_cast<const void *>(a0), nb, fbar);
        }
        const uint32_t tx = __reduce_add_sync(0xffffffffu, nb);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(fbar, tx);
    };

    const int jfirst = min(D, nchunk);
    for (int j = 0; j < jfirst; ++j) issue(j);
    if (tid < NCW * 2) bsum[tid * PAIR_BND] = __int_as_float(-1);
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {
            griddep_wait();
            const int rows = ntask > 0 ? job.ntok : 0;
            const uint32_t bytes = (uint32_t)(tpr * TL::STRIDE);
            for (int r = 0; r < rows; ++r)
                bulk_g2s(xa + (uint32_t)r * tok_stride,
                         job.ximg + (size_t)r * job.ximg_pitch + (size_t)t0 * TL::STRIDE, bytes, xbar);
            mbar_arrive_expect_tx(xbar, bytes * (uint32_t)rows);
        }
        __syncwarp();
    }

    // ---------------------------------------------------------------------- consume
    const int pa0 = (int)tpr_div.div((uint32_t)a);
    const bool a_mid = a < b && a != pa0 * tpr;
    const int ntok = job.ntok;
    mbar_wait(xbar, 0);

    auto store_pair = [&](int p, int m, float v0, float v1) {
        const int r0 = 2 * (p0 + p);
        out[(long)m * N + r0] = v0;
        if (r0 + 1 < N) out[(long)m * N + r0 + 1] = v1;
    };

    float carry[2][MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) carry[0][m] = carry[1][m] = 0.0f;
    int carry_p = -1;

    for (int j = 0; j < nchunk; ++j) {
        const int slot = (j % D) * NCW + warp;
        const int fa = a + j * job.tps;
        mbar_wait(full_bar(slot), (uint32_t)((j / D) & 1));
        const int fb = min(b, fa + job.tps);
        const int f = fa + lane;
        const bool valid = f < fb;
        int p = 0x7fffffff, c = 0;
        uint32_t w0[F::WW], w1[F::WW];
        uint32_t al0 = 0, al1 = 0;
        SAddr xbase = smem;
        if (valid) {
            const int pa = (int)tpr_div.div((uint32_t)fa), ca = fa - pa * tpr;
            const int pb = (int)tpr_div.div((uint32_t)(fb - 1));
            p = (int)tpr_div.div((uint32_t)f);
            c = f - p * tpr;
            SAddr addr0, addr1;
            if (split) {
                // (a stage over more than 4 pairs was flagged when it was issued; its extra
                // lanes read the last run, inside the slot)
                const int k = min(2 * (p - pa), PAIR_RUNS_SPLIT - 2);
                const uint32_t cofs = (uint32_t)(c - (p == pa ? ca : 0)) * TB;
                addr0 = smem + (lds32(hdr(slot, k)) - ring) + cofs;
                addr1 = 2 * (p0 + p) + 1 >= N ? addr0 : smem + (lds32(hdr(slot, k + 1)) - ring) + cofs;
            } else {
                const SAddr h0 = smem + (lds32(hdr(slot, 0)) - ring);
                const SAddr h1 = smem + (lds32(hdr(slot, 1)) - ring);
                const int ra = 2 * pa, r0 = 2 * p;  // CTA-relative rows
                addr0 = p == pa ? h0 + (uint32_t)(c - ca) * TB : h1 + (uint32_t)((r0 - ra - 1) * tpr + c - ca) * TB;
                if (2 * (p0 + p) + 1 >= N)
                    addr1 = addr0;  // the last row of an odd N has no partner
                else if (pb > pa && p == pb)
                    addr1 = smem + (lds32(hdr(slot, 2)) - ring) + (uint32_t)c * TB;
                else
                    addr1 = h1 + (uint32_t)((r0 - ra) * tpr + c - ca) * TB;
            }
            F::load(addr0, w0);
            F::load(addr1, w1);
            al0 = (uint32_t)((uintptr_t)addr0 & 3u);
            al1 = (uint32_t)((uintptr_t)addr1 & 3u);
            xbase = smem + (xa - ring) + (uint32_t)(c * TL::STRIDE);
        }
        __syncwarp();
        if (j + D < nchunk) {
            fence_proxy_async_smem();
            issue(j + D);
        }
        if (fa < fb) {
            PairSink<MT> sink;
#pragma unroll
            for (int m = 0; m < MT; ++m) sink.acc[0][m] = sink.acc[1][m] = 0.0f;
            if (valid) F::compute_pair(w0, al0, w1, al1, XT{xbase, tok_stride}, ntok, sink);
            // segmented reduction: pairs are contiguous runs of lanes
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int p2 = __shfl_down_sync(0xffffffffu, p, d);
                const bool take = lane + d < 32 && p2 == p;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float v = __shfl_down_sync(0xffffffffu, sink.acc[r][m], d);
                        if (take) sink.acc[r][m] += v;
                    }
                }
            }
            const int pprev = __shfl_up_sync(0xffffffffu, p, 1);
            const bool head = valid && (lane == 0 || pprev != p);
            if (head && p == carry_p) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    sink.acc[0][m] += carry[0][m];
                    sink.acc[1][m] += carry[1][m];
                }
            }
            const int flast = min(fb, fa + 32) - 1;
            const int plast = __shfl_sync(0xffffffffu, p, flast - fa);
            const bool cont = (plast + 1) * tpr > flast + 1;
            if (head && !(p == plast && cont)) {
                if (a_mid && p == pa0) {
                    float *e = bsum + (warp * 2) * PAIR_BND;  // shared with the previous warp
                    e[0] = __int_as_float(p);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        e[1 + m] = sink.acc[0][m];
                        e[17 + m] = sink.acc[1][m];
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < ntok) store_pair(p, m, sink.acc[0][m], sink.acc[1][m]);
                }
            }
            const int hl = __reduce_min_sync(0xffffffffu, (valid && p == plast) ? lane : 31);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                carry[0][m] = __shfl_sync(0xffffffffu, sink.acc[0][m], hl);
                carry[1][m] = __shfl_sync(0xffffffffu, sink.acc[1][m], hl);
            }
            carry_p = cont ? plast : -1;
        }
    }
    // as in engine_kernel: this warp's copies still in flight land before the CTA exits
    if (lane == 0) {
        for (int d = 0; d < D && d < nchunk; ++d)
            mbar_drain(full_bar(d * NCW + warp), (uint32_t)(((d + D * ((nchunk - 1 - d) / D)) / D) & 1), DRAIN_NS);
        if (warp == 0) mbar_drain(xbar, 0, DRAIN_NS);
    }
    // a range that ended inside a pair: its sums are shared with the next warp
    if (carry_p >= 0 && lane == 0) {
        float *e = bsum + (warp * 2 + ((a_mid && carry_p == pa0) ? 0 : 1)) * PAIR_BND;
        e[0] = __int_as_float(carry_p);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            e[1 + m] = carry[0][m];
            e[17 + m] = carry[1][m];
        }
    }
    consumer_sync<NCONS>();
    // pairs shared by consecutive warps: their sums added in warp order (lane m: token m)
    if (warp == 0) {
        int cur = -1;
        float acc0 = 0.0f, acc1 = 0.0f;
        for (int w = 0; w < NCW; ++w) {
            for (int side = 0; side < 2; ++side) {
                const float *e = bsum + (w * 2 + side) * PAIR_BND;
                const int r = __float_as_int(e[0]);
                if (r < 0) continue;
                if (r != cur) {
                    if (cur >= 0 && lane < ntok) store_pair(cur, lane, acc0, acc1);
                    cur = r;
                    acc0 = acc1 = 0.0f;
                }
                if (lane < ntok) {
                    acc0 += e[1 + lane];
                    acc1 += e[17 + lane];
                }
            }
        }
        if (cur >= 0 && lane < ntok) store_pair(cur, lane, acc0, acc1);
    }
}

}  // namespace qg
