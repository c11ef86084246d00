// qg_plan.h -- host-side launch planning shared by the workspace query and the launchers.
//
// Everything here is a pure function of the problem shape and the device's SM count, so
// qg_workspace_size() and the launchers always agree.  The split-K factor depends on the
// shape only (never on the device).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <algorithm>

#include "qg_engine.cuh"
#include "qg_engine1.cuh"
#include "qg_prefill.cuh"

namespace qg {

struct FmtInfo {
    int qk, bs;
};

inline bool fmt_info(int fmt, FmtInfo &f) {
    switch (fmt) {
    case 2: f = {32, 18}; return true;     // Q4_0
    case 3: f = {32, 20}; return true;     // Q4_1
    case 6: f = {32, 22}; return true;     // Q5_0
    case 7: f = {32, 24}; return true;     // Q5_1
    case 20: f = {32, 18}; return true;    // IQ4_NL
    case 8: f = {32, 34}; return true;     // Q8_0
    case 10: f = {256, 84}; return true;   // Q2_K
    case 11: f = {256, 110}; return true;  // Q3_K
    case 12: f = {256, 144}; return true;  // Q4_K
    case 13: f = {256, 176}; return true;  // Q5_K
    case 14: f = {256, 210}; return true;  // Q6_K
    case 23: f = {256, 136}; return true;  // IQ4_XS
    default: return false;
    }
}

constexpr int G_PLAN = 152;               // split-K planning constant
constexpr uint32_t XCAP = 140 * 1024;     // activation tiles held by one CTA
constexpr int DMAX = 4;                   // ring slots per consumer warp
constexpr int M_MAX = 16;
constexpr int XREP = 31;  // repeated activation tiles past a row's end (a stage's 32 lanes)

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int pick_mt(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }
inline int log2i(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

// Task geometry of a row of K elements (must match the format traits in qg_formats.cuh):
//   Q4_0, IQ4_NL: 16 (only with long_tasks), 8, 4 or 1 blocks per task; Q4_1,
//   Q5_0, Q5_1, Q8_0: 8 (only with long_tasks), 4 or 1; Q2_K, Q4_K, IQ4_XS: 2 or 1
//   superblocks (the largest that divides the row); Q3_K, Q5_K, Q6_K: one whole superblock.
// long_tasks asks for 16-block Q4_0 and IQ4_NL tasks (288 bytes, the size of two Q4_K superblocks): with
// one token per lane they leave the lane's decode fewer, longer loads and let the 12-warp
// engine run; with several tokens per lane the 8-block tasks on 16 warps were faster.  It
// also asks for 8-block Q5_0 and Q8_0 tasks (176 and 272 bytes, multiples of 16 where their
// 4-block tasks of 88 and 136 bytes are not) and 8-block Q4_1 and Q5_1 tasks (160 and 192
// bytes: fewer, longer tasks per lane).
struct TaskGeo {
    bool ok = false;
    int T = 1, TPB = 1, BPT = 1, XGT = 8, nbr = 0, gpr = 0, tpr = 0, stride = 0, bs = 0;
    uint32_t rb = 0;
    uint32_t bytes_of(int ntask) const { return (uint32_t)(((ntask + TPB - 1) / TPB) * BPT * bs); }
    int task_bytes() const { return BPT * bs / TPB; }
    // every task of every row starts 16-byte aligned (rows start at multiples of rb from a
    // 16-byte-aligned tensor): runs need no widening
    bool aligned16() const { return task_bytes() % 16 == 0 && rb % 16 == 0; }
    // every stage of the one-token engines is a 16-byte-aligned bulk copy: CTA row ranges cut
    // at multiples of row_align_unit(rb) rows, task ranges at multiples of task_align_unit
    // tasks (both at most 8 for even sizes)
    bool stage_aligned() const { return TPB == 1 && task_bytes() % 2 == 0 && rb % 2 == 0; }
};
inline TaskGeo task_geo(int fmt, int K, bool long_tasks) {
    TaskGeo g;
    FmtInfo f;
    if (!fmt_info(fmt, f) || K < f.qk || K % f.qk) return g;
    g.bs = f.bs;
    g.nbr = K / f.qk;
    g.rb = (uint32_t)(g.nbr * f.bs);
    if (f.qk == 32) {
        g.T = (long_tasks && (fmt == 2 || fmt == 20) && g.nbr % 16 == 0)   ? 16
              : ((fmt == 2 || fmt == 20) && g.nbr % 8 == 0)                ? 8
              : (long_tasks && (fmt == 3 || fmt == 6 || fmt == 7 || fmt == 8) && g.nbr % 8 == 0) ? 8
              : g.nbr % 4 == 0                                             ? 4
                                                                           : 1;
        g.BPT = g.T;
        g.XGT = g.T;
        g.TPB = 1;
        g.gpr = g.nbr / g.T;
    } else if (fmt == 11 || fmt == 13 || fmt == 14) {
        g.T = 2;
        g.BPT = 1;
        g.TPB = 1;
        g.XGT = 8;
        g.gpr = g.nbr;
    } else {
        g.T = g.nbr % 2 == 0 ? 2 : 1;
        g.BPT = g.T;
        g.TPB = 1;
        g.XGT = 8 * g.T;
        g.gpr = g.nbr / g.T;
    }
    g.tpr = g.gpr * g.TPB;
    g.stride = tile_stride(g.XGT);
    g.ok = true;
    return g;
}
inline int geo_ncw(const TaskGeo &g, int MT) { return engine_ncw(g.task_bytes(), MT); }

// The rows of task_geo cut into one-superblock tasks where task_geo pairs superblocks (Q2_K,
// Q4_K, IQ4_XS with an even superblock count): twice the tasks, each half the decode chain,
// and 16 warps instead of 8 where the task drops to 160 bytes or less.  For launches whose
// CTAs have too few tasks to keep 8 warps' decode chains overlapped.
inline TaskGeo short_task_geo(int fmt, int K) {
    TaskGeo g = task_geo(fmt, K, false);
    if (!g.ok || g.T != 2 || g.BPT != 2) return g;
    g.T = 1;
    g.BPT = 1;
    g.XGT = 8;
    g.gpr = g.nbr;
    g.tpr = g.gpr * g.TPB;
    g.stride = tile_stride(g.XGT);
    return g;
}

// Geometry of one row's part of a row-pair task (engine_pair_kernel): one Q4_K, Q5_K, Q6_K
// or IQ4_XS superblock, eight Q4_0 or IQ4_NL blocks, or four Q8_0 / Q4_1 / Q5_0 / Q5_1
// blocks (rows whose block count is a multiple of that); not ok otherwise (Q2_K and Q3_K,
// whose decode outweighs their activation traffic, measured no gain from pairs).
inline TaskGeo pair_geo(int fmt, int K) {
    TaskGeo g = task_geo(fmt, K, false);
    if (!g.ok) return g;
    if (fmt == 12 || fmt == 23) {  // Q4_K, IQ4_XS
        g.T = 1, g.BPT = 1, g.XGT = 8, g.gpr = g.nbr;
    } else if (fmt == 13 || fmt == 14) {  // Q5_K, Q6_K
        g.T = 2, g.BPT = 1, g.XGT = 8, g.gpr = g.nbr;  // the whole-superblock task of these formats
    } else if ((fmt == 2 || fmt == 20) && g.nbr % 8 == 0) {
        g.T = 8, g.BPT = 8, g.XGT = 8, g.gpr = g.nbr / 8;
    } else if ((fmt == 8 || fmt == 3 || fmt == 6 || fmt == 7) && g.nbr % 4 == 0) {
        g.T = 4, g.BPT = 4, g.XGT = 4, g.gpr = g.nbr / 4;
    } else {
        g.ok = false;
        return g;
    }
    g.tpr = g.gpr;
    g.stride = tile_stride(g.XGT);
    return g;
}
// Warps of a launch whose CTAs hold up to tasks_per_cta tasks.
inline int plan_ncw(const TaskGeo &g, int MT, long tasks_per_cta) {
    if (ncw_wide_allowed(g.task_bytes(), MT) && tasks_per_cta >= (long)NCW_WIDE * 32 * 2) return NCW_WIDE;
    return geo_ncw(g, MT);
}

// Stage size and ring of one engine launch.
struct Ring {
    bool ok = false;
    int tps = 0, depth = 0;
    uint32_t slot_bytes = 0, x_bytes = 0, j_bytes = 0, smem_total = 0;
};
// run: the fewest tasks in one run of adjacent rows that any CTA of the launch sees (0: the
// whole CTA range is one run); a stage of t tasks then spans at most t / run + 2 runs.
// ncw: warps of the launch (geo_ncw).
// tasks_per_cta (0: unknown): the most tasks one CTA of the launch holds; the ring then has
// no more slots per warp than a warp has stages, so that a CTA with little work keeps its
// shared memory small and the next kernel's CTAs can be resident beside it.
inline Ring plan_ring(const TaskGeo &g, long run, uint32_t x_bytes, uint32_t j_bytes, int ncw, long tasks_per_cta = 0) {
    Ring r;
    r.x_bytes = (uint32_t)align_up(x_bytes, 16);
    r.j_bytes = (uint32_t)align_up(j_bytes, 16);
    const long avail = (long)SMEM_MAX - (long)engine_fixed_smem(ncw * DMAX, ncw) - (long)r.x_bytes - (long)r.j_bytes;
    // a stage is one task per lane (fewer only when not even one slot per warp would fit)
    for (int tps = 32; tps >= 2; tps /= 2) {
        int t = tps;
        int pieces = 1;
        if (run > 0) {
            t = (int)std::min<long>(t, (long)(NPIECE_MAX - 2) * run);
            t = std::max(2, t / 2 * 2);
            pieces = (int)std::min<long>(NPIECE_MAX, ((long)t + run - 1) / run + 1);
            if ((long)t > (long)(NPIECE_MAX - 1) * run) return r;  // runs too short for the piece table
        }
        const uint32_t slot = (uint32_t)align_up(g.bytes_of(t) + 32u * pieces, 16);
        const long d = avail / ((long)ncw * (slot + STAGE_SLACK));
        if (d >= 1) {
            r.tps = t;
            r.slot_bytes = slot;
            r.depth = (int)std::min<long>(DMAX, d);
            if (tasks_per_cta > 0) {
                // a warp's tasks are whole units of TPB: at most ceil(units / ncw) units
                const long per_warp = ((tasks_per_cta + g.TPB - 1) / g.TPB + ncw - 1) / ncw * g.TPB;
                r.depth = (int)std::min<long>(r.depth, std::max<long>(1, (per_warp + t - 1) / t));
            }
            break;
        }
    }
    if (r.depth < 1) return r;
    const int S = ncw * r.depth;
    r.smem_total = (uint32_t)S * (r.slot_bytes + STAGE_SLACK) + r.x_bytes + r.j_bytes + engine_fixed_smem(S, ncw);
    r.ok = r.smem_total <= (uint32_t)SMEM_MAX;
    return r;
}

// Ring of a row-pair launch: stages of 32 two-row tasks, at most PAIR_RUNS runs each (whole
// rows) or PAIR_RUNS_SPLIT (K-slices).
inline Ring plan_ring_pair(const TaskGeo &g, uint32_t x_bytes, int ncw, bool split = false) {
    Ring r;
    r.x_bytes = (uint32_t)align_up(x_bytes, 16);
    const long avail = (long)SMEM_MAX - (long)pair_fixed_smem(ncw * DMAX, ncw) - (long)r.x_bytes;
    const uint32_t slot = (uint32_t)align_up(
        2u * g.bytes_of(32) + (g.aligned16() ? 0u : 32u * (split ? PAIR_RUNS_SPLIT : PAIR_RUNS)), 16);
    const long d = avail / ((long)ncw * (slot + STAGE_SLACK));
    if (d < 1) return r;
    r.tps = 32;
    r.slot_bytes = slot;
    r.depth = (int)std::min<long>(DMAX, d);
    const int S = ncw * r.depth;
    r.smem_total = (uint32_t)S * (r.slot_bytes + STAGE_SLACK) + r.x_bytes + pair_fixed_smem(S, ncw);
    r.ok = r.smem_total <= (uint32_t)SMEM_MAX;
    return r;
}

// ----------------------------------------------------------------------------- GEMV
struct GemvPlan {
    bool ok = false;
    TaskGeo geo;
    int KS = 1, groups = 1, grid = 1, MT = 1, tpr_x = 0, ncw = 8;
    bool pair = false;  // row-pair engine: tasks of two rows (engine_pair_kernel)
    int MC = 0;         // row pairs: tokens per launch (launches over token chunks of MC)
    int xrep = 0;       // one-row engine: activation tiles repeated past a row's end
    Ring ring;
    // one-token engine for 16-byte-aligned rows (engine1_kernel): ncw warps, depth slots each
    bool one = false;
    int one_depth = 0;
    uint32_t one_slot = 0, one_x = 0, one_smem = 0;
    size_t ws_ximg = 0, ximg_pitch = 0, ws_part = 0, ws_total = 0;
};

// Partial sums of one CTA of the one-token engine (rows x tasks per row) at most this many.
constexpr int ONE_PART_MAX = 8192;
// Tasks that are not a multiple of 16 bytes (Q6_K, Q3_K and Q2_K superblocks, short legacy
// groups) take the one-token engine only where a CTA streams at least this many bytes:
// measured slower than the general engine at 4096 x 4096 (Q2_K, Q3_K: 36, 47 KB per CTA),
// faster from 17408 x 5120 (190-480 KB per CTA).
constexpr long ONE_UNALIGNED_MIN_BYTES = 128 * 1024;
// Rows up to this length are quantized inside the one-token engine (every CTA quantizes the
// whole row, a cost that grows with K; beyond this the preparation kernel and its extra
// kernel boundary were measured faster).
constexpr int ONE_FUSED_K_MAX = 8192;

// The one-token engine where it applies: one token, no K-split, every task and row a
// multiple of 16 bytes (so each stage is one aligned bulk copy), and the CTA's partial sums
// within ONE_PART_MAX.  Warps as the general engine (plan_ncw): 16 for tasks of at most 160
// bytes, else 12 where every warp gets at least two stages and 8 otherwise; as many ring
// slots per warp (up to DMAX) as shared memory holds.
inline void plan_gemv_one(GemvPlan &p, int N, int sms) {
    const TaskGeo &g = p.geo;
    if (p.pair || p.MT != 1 || p.KS != 1 || !g.stage_aligned()) return;
    const int ra = row_align_unit(g.rb);
    if (N % ra) return;
    const int grid = std::min(N / ra, sms);
    const long rows_max = (long)ra * ((N / ra + grid - 1) / grid);
    if (g.task_bytes() % 16 != 0 && rows_max * (long)g.rb < ONE_UNALIGNED_MIN_BYTES) return;
    const long part = rows_max * g.tpr;
    if (part > ONE_PART_MAX) return;
    // the general engine's warp count: 12 only where every warp gets two stages or more
    const int ncw = plan_ncw(g, 1, part);
    const uint32_t slot = (uint32_t)(32 * g.task_bytes());
    const uint32_t xb = (uint32_t)align_up((size_t)(g.tpr + XREP) * g.stride, 16);
    int depth = 0;
    for (int d = DMAX; d >= 1; --d)
        if (engine1_smem(ncw * d, slot, xb, (int)part) <= (uint32_t)SMEM_MAX) {
            depth = d;
            break;
        }
    if (depth < 1) return;
    p.one = true;
    p.ncw = ncw;
    p.grid = grid;
    p.groups = grid;
    p.tpr_x = g.tpr;
    p.xrep = XREP;
    p.one_depth = depth;
    p.one_slot = slot;
    p.one_x = xb;
    p.one_smem = engine1_smem(ncw * depth, slot, xb, (int)part);
}

// long_ok: one token may take the long tasks of task_geo
inline GemvPlan plan_gemv(int fmt, int N, int K, int M, int sms, bool long_ok = true) {
    GemvPlan p;
    p.geo = task_geo(fmt, K, long_ok && pick_mt(M) == 1);
    const TaskGeo &g = p.geo;
    if (!g.ok || N < 1 || M < 1 || M > M_MAX || sms < 1) return p;
    p.KS = N < G_PLAN / 2 ? std::min(g.gpr, (G_PLAN + N - 1) / N) : 1;
    const bool split_for_n = p.KS > 1;
    auto xbytes = [&](int ks) { return (long)M * ((g.gpr + ks - 1) / ks) * g.TPB * g.stride; };
    while (xbytes(p.KS) > (long)XCAP && p.KS < g.gpr) ++p.KS;
    if (xbytes(p.KS) > (long)XCAP) return p;
    p.groups = std::min(N, std::max(1, sms / p.KS));
    p.grid = p.groups * p.KS;
    p.MT = pick_mt(M);
    p.tpr_x = (g.gpr + p.KS - 1) / p.KS * g.TPB;
    // split-K: every row is its own run; the shortest slice has floor(gpr / KS) groups
    p.ncw = plan_ncw(g, p.MT, (long)((N + p.groups - 1) / p.groups) * p.tpr_x);
    // one token: every row's tiles are followed by copies of its first XREP tiles, so that
    // the 32 lanes of a stage read consecutive tiles even where the stage wraps to the next
    // row (no bank conflicts between a row's last tiles and the next row's first)
    const long xrep_bytes = (long)M * (p.tpr_x + XREP) * g.stride;
    p.xrep = (p.MT == 1 && xrep_bytes <= (long)XCAP) ? XREP : 0;
    p.ring = plan_ring(g, p.KS == 1 ? 0 : (long)(g.gpr / p.KS) * g.TPB,
                       (uint32_t)((long)M * (p.tpr_x + p.xrep) * g.stride), 0, p.ncw);
    if (!p.ring.ok) return p;
    // row pairs: a GEMV of whole rows (not split for lack of rows) with at least two rows
    // and two tokens (with one token the one-row tasks measured faster).  When the tiles of
    // all tokens do not fit, the tokens go in chunks of MC, the largest power of two whose
    // tiles do (each chunk streams the weights again: measured faster than the split-K
    // one-row launch at 8 and 16 tokens on rows of 17408).
    if (!split_for_n && N >= 2 && p.MT >= 2) {
        const TaskGeo pg = pair_geo(fmt, K);
        // Q5_K / Q6_K pairs hold 88 / 108 words of weights: at 16 tokens per lane they ran
        // out of registers, so they take at most 8 tokens per launch (two launches of 8
        // measured faster than one one-row launch of 16)
        int mc = (fmt == 13 || fmt == 14) ? std::min(M, 8) : M;
        // tiles of mc tokens over a 1/ks slice of the row; slices keep at least
        // PAIR_SPLIT_MIN_TPR tasks and every slice group at least 16 CTAs
        auto slice_x = [&](int m, int ks) { return (long)m * ((pg.gpr + ks - 1) / ks) * pg.stride; };
        auto ks_ok = [&](int ks) { return ks == 1 || (pg.gpr / ks >= PAIR_SPLIT_MIN_TPR && sms / ks >= 16); };
        int ks = 1;
        while (pg.ok && mc >= 2) {
            ks = 1;
            while (slice_x(mc, ks) > (long)XCAP && ks_ok(ks + 1)) ++ks;
            if (slice_x(mc, ks) <= (long)XCAP) break;
            mc = pick_mt(mc) / 2;  // tokens in chunks instead
        }
        const int mt = pick_mt(mc) < 2 ? 2 : pick_mt(mc);
        if (pg.ok && mc >= 1 && slice_x(mc, ks) <= (long)XCAP) {
            const int P = (N + 1) / 2, pgroups = std::min(P, sms / ks);
            const int pncw = 8;  // two-row tasks of 288 to 420 bytes and two or more tokens per lane
            const Ring pr = plan_ring_pair(pg, (uint32_t)slice_x(mc, ks), pncw, ks > 1);
            if (pr.ok) {
                p.pair = true;
                p.geo = pg;
                p.KS = ks;
                p.MT = mt;
                p.MC = mc;
                p.groups = pgroups;
                p.grid = pgroups * ks;
                p.tpr_x = (pg.gpr + ks - 1) / ks;
                p.ncw = pncw;
                p.ring = pr;
            }
        }
    }
    plan_gemv_one(p, N, sms);
    size_t o = 0;
    p.ximg_pitch = (size_t)g.tpr * g.stride;
    p.ws_ximg = o;
    o = align_up(o + p.ximg_pitch * M, 256);
    if (p.KS > 1) {
        p.ws_part = o;
        o = align_up(o + 4ull * p.KS * M * N, 256);
    }
    p.ws_total = o;
    p.ok = true;
    return p;
}

// ----------------------------------------------------------------------------- FFN sublayer
struct FfnPlan {
    bool ok = false;
    TaskGeo geo;
    int grid = 1, MT = 1, MC = 1, nchunk = 1, ncw = 8;
    Ring ring;
    GemvPlan gate;  // several tokens: gate and up as two row-pair GEMV launches (gate.pair)
    GemvPlan down;  // y = Wd h; h = silu(g) * u is formed by its activation preparation
    // one token: gate/up on the one-token engine with SwiGLU and the requantization of h in
    // its epilogue (ffn_gateup1_kernel), writing the down projection's tile image
    bool one = false;
    int one_grid = 0, one_ncw = 0, one_depth = 0;
    uint32_t one_slot = 0, one_x = 0, one_smem = 0;
    size_t ws_ximg = 0, ximg_pitch = 0, ws_g = 0, ws_u = 0, ws_h = 0, ws_down = 0, ws_total = 0;
};

inline FfnPlan plan_ffn(int fmt, int M, int H, int I, int sms) {
    FfnPlan p;
    // IQ4_NL in 8-block tasks here: with 16-block tasks (gate/up, down or both) the sublayer
    // measured 1.4-1.7 us slower at H = 5120, I = 17408 (register spills), although the plain
    // GEMV gains from them
    p.geo = task_geo(fmt, H, M == 1 && fmt != 20);
    const TaskGeo &g = p.geo;
    if (!g.ok || !task_geo(fmt, I, false).ok || M < 1 || M > M_MAX || sms < 1) return p;
    const long tiles = (long)g.tpr * g.stride;
    p.MC = (int)std::min<long>(M, (long)XCAP / tiles);
    if (p.MC < 1) return p;
    p.nchunk = (M + p.MC - 1) / p.MC;
    p.MT = pick_mt(p.MC);
    p.grid = std::min(2 * I, sms);
    p.ncw = plan_ncw(g, p.MT, (long)((2L * I + p.grid - 1) / p.grid) * g.tpr);
    p.ring = plan_ring(g, (long)I * g.tpr, (uint32_t)(p.MC * tiles), 0, p.ncw);
    if (!p.ring.ok) return p;
    p.down = plan_gemv(fmt, H, I, M, sms, fmt != 20);
    if (!p.down.ok) return p;
    if (M >= 2) p.gate = plan_gemv(fmt, I, H, M, sms);
    if (p.gate.pair && p.gate.KS > 1) p.gate.pair = false;  // its partial sums have no workspace here
    if (M == 1 && p.down.one && g.stage_aligned() && I % 32 == 0) {
        // every CTA the same number of units (nu): the launch takes as long as its fullest CTA
        const int U = I / 32, nu = (U + std::min(U, sms) - 1) / std::min(U, sms), grid = (U + nu - 1) / nu;
        const int part = ffn1_part_floats(nu, g.tpr);
        const int ncw = plan_ncw(g, 1, 64L * nu * g.tpr);
        const uint32_t slot = (uint32_t)(32 * g.task_bytes());
        const uint32_t xb = (uint32_t)align_up((size_t)(g.tpr + XREP) * g.stride, 16);
        for (int d = DMAX; d >= 1 && !p.one; --d) {
            const uint32_t sm = engine1_smem(ncw * d, slot, xb, part);
            if (part <= 4 * ONE_PART_MAX && sm <= (uint32_t)SMEM_MAX) {
                p.one = true;
                p.one_grid = grid;
                p.one_ncw = ncw;
                p.one_depth = d;
                p.one_slot = slot;
                p.one_x = xb;
                p.one_smem = sm;
            }
        }
    }
    size_t o = 0;
    p.ximg_pitch = (size_t)(p.gate.pair ? p.gate.ximg_pitch : tiles);
    p.ws_ximg = o; o = align_up(o + p.ximg_pitch * M, 256);
    p.ws_g = o; o = align_up(o + 4ull * M * I, 256);
    p.ws_u = o; o = align_up(o + 4ull * M * I, 256);
    p.ws_h = o; o = align_up(o + 4ull * M * I, 256);
    p.ws_down = o;
    o = align_up(o + p.down.ws_total, 256);
    p.ws_total = o;
    p.ok = true;
    return p;
}

// ----------------------------------------------------------------------------- MoE FFN
struct MoePlan {
    bool ok = false;
    int S = 0, P = 1, gu_ncw = 8, dn_ncw = 8;  // P: activation rows per token (s16: 2 planes)
    TaskGeo gh, gi;  // rows of H elements (gate/up) and of I elements (down)
    int gu_grid = 0, dn_grid = 0, dn_MC = 1, dn_nchunk = 1;
    Ring gu_ring, dn_ring;
    size_t ws_g = 0, ws_u = 0, ws_h = 0, ws_hq = 0, ws_hd = 0, ws_hs = 0, ws_logits = 0, ws_ids = 0, ws_w = 0,
           ws_ximg = 0, ws_himg = 0, ximg_pitch = 0, himg_pitch = 0, ws_total = 0;
};

inline MoePlan plan_moe(int fmt, int M, int H, int E, int topk, int I, int sms, bool s16 = false) {
    MoePlan p;
    p.P = s16 ? 2 : 1;
    // one-superblock tasks: an expert's rows are few per CTA at every batch size (measured
    // faster than superblock pairs from 1 to 16 tokens)
    p.gh = short_task_geo(fmt, H);
    p.gi = short_task_geo(fmt, I);
    if (!p.gh.ok || !p.gi.ok || M < 1 || M > M_MAX || E < 1 || E > 1024 || topk < 1 || topk > 16 || topk > E ||
        sms < 1 || M * topk > SCRATCH_W)
        return p;
    p.S = topk + 1;
    // gate/up: units of 32 positions j of one (token, slot), each its 32 gate and 32 up rows;
    // a CTA holds the g and u of its units (P planes each) for the requantization of h
    const long gu_units = (long)M * p.S * (I / 32);
    const long gu_x = (long)M * p.P * p.gh.tpr * p.gh.stride;
    if (gu_x > (long)XCAP) return p;
    p.gu_grid = (int)std::min<long>(sms, gu_units);
    const long upc = (gu_units + p.gu_grid - 1) / p.gu_grid;  // most units of one CTA
    p.gu_ncw = plan_ncw(p.gh, p.P, upc * 64 * p.gh.tpr);
    p.gu_ring = plan_ring(p.gh, 32L * p.gh.tpr, (uint32_t)gu_x, (uint32_t)(upc * 64 * p.P * 4), p.gu_ncw,
                          upc * 64 * p.gh.tpr);
    if (!p.gu_ring.ok) return p;
    // down: per CTA a range of hidden rows; output rows (token, slot, row) in shared memory
    const long tiles_tok = (long)p.S * p.P * p.gi.tpr * p.gi.stride;
    p.dn_grid = std::min(sms, H);
    const int nloc = (H + p.dn_grid - 1) / p.dn_grid;
    const long part_tok = 4L * p.S * p.P * nloc;
    p.dn_MC = (int)std::min<long>(M, (long)XCAP / (tiles_tok + part_tok));
    if (p.dn_MC < 1) return p;
    p.dn_nchunk = (M + p.dn_MC - 1) / p.dn_MC;
    // CTAs own floor or ceil of H / dn_grid rows: runs are at least the floor long
    p.dn_ncw = geo_ncw(p.gi, p.P);
    p.dn_ring = plan_ring(p.gi, (long)(H / p.dn_grid) * p.gi.tpr, (uint32_t)(p.dn_MC * tiles_tok),
                          (uint32_t)(p.dn_MC * part_tok), p.dn_ncw, (long)p.dn_MC * p.S * nloc * p.gi.tpr);
    if (!p.dn_ring.ok) return p;
    // workspace
    const size_t Rw = (size_t)M * p.S;
    size_t o = 0;
    p.ws_g = o; o = align_up(o + 4 * Rw * p.P * I, 256);   // [token][slot][plane][I]
    p.ws_u = o; o = align_up(o + 4 * Rw * p.P * I, 256);
    p.ws_h = o; o = align_up(o + 4 * Rw * I, 256);
    p.ws_hq = o; o = align_up(o + Rw * p.P * I, 256);        // int8, or int16 codes for s16
    p.ws_hd = o; o = align_up(o + 4 * Rw * (I / 32), 256);
    p.ws_hs = o; o = align_up(o + 4 * Rw * (I / 32), 256);
    p.ws_logits = o; o = align_up(o + 4ull * M * E, 256);
    p.ws_ids = o; o = align_up(o + 4ull * M * topk, 256);
    p.ws_w = o; o = align_up(o + 4ull * M * topk, 256);
    p.ximg_pitch = (size_t)p.gh.tpr * p.gh.stride;
    p.himg_pitch = (size_t)p.gi.tpr * p.gi.stride;
    p.ws_ximg = o; o = align_up(o + p.ximg_pitch * M * p.P, 256);
    p.ws_himg = o; o = align_up(o + p.himg_pitch * Rw * p.P, 256);
    p.ws_total = o;
    p.ok = true;
    return p;
}

// ----------------------------------------------------------------------------- prefill GEMM
// Tiles of 128 weight rows x NT token tiles of BT tokens (BT = 256, or M rounded up to 16 when
// M < 256; NT = 1 or 2) over K-slices of whole 64-element K tiles.  NT and the slice count KS
// minimise an estimate of the critical path in K-tile times of one token tile: (waves of CTAs
// over the SMs) x (K tiles per CTA) x max(NT, 1.5) -- a K tile's dequantization costs about
// 1.5 MMA steps of one token tile and overlaps them -- plus for KS > 1 the partial sums'
// traffic (KS x M x N x 8 bytes at about 6 TB/s; one K-tile time is 2 x 128 x BT x 64 flops
// at 1/SM of about 1.8 PFLOP/s).
struct PrefillPlan {
    bool ok = false;
    int BT = 0, NT = 1, ntt = 0, ngrp = 0, nn = 0, nkt = 0, KS = 1, ktps = 0, stages = 0, tmem_cols = 0;
    uint32_t rb = 0, smem = 0, idesc = 0;
    size_t ws_ximg = 0, ws_part = 0, ws_total = 0;
};

constexpr int PF_M_MAX = 1 << 20;

inline PrefillPlan plan_prefill(int fmt, int N, int K, int M, int sms) {
    PrefillPlan p;
    FmtInfo f;
    if (!fmt_info(fmt, f) || K < f.qk || K % f.qk || N < 1 || M < 1 || M > PF_M_MAX || sms < 1) return p;
    p.rb = (uint32_t)((K / f.qk) * f.bs);
    p.BT = M >= PF_MAX_BT ? PF_MAX_BT : (M + 15) / 16 * 16;
    p.ntt = (M + p.BT - 1) / p.BT;
    p.nn = (N + PF_BM - 1) / PF_BM;
    p.nkt = (K + PF_BK - 1) / PF_BK;
    const double ktile_s = 2.0 * PF_BM * p.BT * PF_BK * sms / 1.8e15;
    const double part_s = (double)M * N * 8.0 / 6.0e12;
    double best = 1e300;
    for (int nt = 1; nt <= 2 && nt <= p.ntt; ++nt) {
        const int ngrp = (p.ntt + nt - 1) / nt;
        for (int ks = 1; ks <= 16 && ks <= p.nkt; ++ks) {
            const int ktps = (p.nkt + ks - 1) / ks;
            const int kse = (p.nkt + ktps - 1) / ktps;  // slices that are not empty
            if (kse != ks) continue;
            if (ks > 1 && ktps < 4) break;
            const long ctas = (long)p.nn * ngrp * ks;
            const long waves = (ctas + sms - 1) / sms;
            const double cost = (double)waves * ktps * std::max(1.5, (double)nt) + (ks > 1 ? ks * part_s / ktile_s : 0.0);
            if (cost < best - 1e-9) {
                best = cost;
                p.NT = nt;
                p.KS = ks;
                p.ktps = ktps;
            }
        }
    }
    if (p.ktps < 1) return p;
    p.ngrp = (p.ntt + p.NT - 1) / p.NT;
    p.stages = 4;
    while (p.stages > 2 && prefill_smem_bytes(p.BT, p.NT, p.stages) > (uint32_t)SMEM_MAX) --p.stages;
    p.smem = prefill_smem_bytes(p.BT, p.NT, p.stages);
    if (p.smem > (uint32_t)SMEM_MAX || !umma_shape_ok(PF_BM, p.BT)) return p;
    p.tmem_cols = tmem_cols_for(p.NT * p.BT);
    p.idesc = umma_idesc_f16(PF_BM, p.BT);
    size_t o = 0;
    p.ws_ximg = o;
    o = align_up(o + (size_t)p.ntt * p.nkt * p.BT * 128, 256);
    if (p.KS > 1) {
        p.ws_part = o;
        o = align_up(o + 4ull * p.KS * M * N, 256);
    }
    p.ws_total = o;
    p.ok = true;
    return p;
}

}  // namespace qg
