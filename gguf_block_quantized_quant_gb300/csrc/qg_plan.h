// qg_plan.h -- host-side launch planning shared by the workspace query and the launchers.
//
// Everything here is a pure function of the problem shape and the device's SM count, so
// qg_workspace_size() and the launchers always agree.  The split-K factor depends on the
// shape only (never on the device), which keeps the order of every floating-point sum
// independent of the GPU the call runs on.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <algorithm>

#include "qg_common.cuh"

namespace qg {

struct FmtInfo {
    int qk, bs, upb;
};

inline bool fmt_info(int fmt, FmtInfo &f) {
    switch (fmt) {
    case 2: f = {32, 18, 1}; return true;     // Q4_0
    case 8: f = {32, 34, 1}; return true;     // Q8_0
    case 12: f = {256, 144, 8}; return true;  // Q4_K
    case 13: f = {256, 176, 8}; return true;  // Q5_K
    case 14: f = {256, 210, 8}; return true;  // Q6_K
    case 23: f = {256, 136, 8}; return true;  // IQ4_XS
    default: return false;
    }
}

constexpr int G_PLAN = 152;                    // split-K planning constant
constexpr uint32_t XSMEM_CAP = 96 * 1024;      // activation codes kept in shared memory
constexpr uint32_t STAGE_TARGET = 32 * 1024;   // bytes of weights per ring slot
constexpr int MAX_SLOTS = 16;
constexpr int M_MAX = 16;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Must match make_xarea() in qg_jobs.cuh.
inline uint32_t xarea_bytes(int rows, int cols) {
    return (uint32_t)(align_up((size_t)rows * cols, 16) + 8ull * rows * (cols / 32));
}
inline int pick_mt(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

// Ring of nslots slots of slot_bytes able to hold stages of up to `stage_bytes`.
struct Ring {
    uint32_t slot_bytes = 0;
    int nslots = 0;
    uint32_t smem_total = 0;
    bool ok = false;
};
inline Ring plan_ring(uint32_t stage_bytes, uint32_t job_smem) {
    Ring r;
    r.slot_bytes = (uint32_t)align_up(stage_bytes + 32, 16);
    const long avail = (long)SMEM_MAX - (long)engine_fixed_smem(MAX_SLOTS) - (long)job_smem;
    if (avail <= 0) return r;
    r.nslots = (int)std::min<long>(MAX_SLOTS, avail / (long)(r.slot_bytes + STAGE_SLACK));
    if (r.nslots < 2) return r;
    r.smem_total = (uint32_t)r.nslots * (r.slot_bytes + STAGE_SLACK) + engine_fixed_smem(r.nslots) + job_smem;
    r.ok = r.smem_total <= (uint32_t)SMEM_MAX;
    return r;
}
// Per-slot byte budget that still leaves room for >= 4 slots.
inline uint32_t stage_budget(uint32_t job_smem) {
    const long avail = (long)SMEM_MAX - (long)engine_fixed_smem(MAX_SLOTS) - (long)job_smem;
    long tb = std::min<long>(STAGE_TARGET, avail / 4 - STAGE_SLACK - 32);
    return tb > 0 ? (uint32_t)(tb / 16 * 16) : 0;
}

// ----------------------------------------------------------------------------- GEMV
struct GemvPlan {
    bool ok = false;
    int nbr = 0, KS = 1, groups = 1, grid = 1, MT = 1, R = 0, segb = 0, kslice_max = 0;
    uint32_t rb = 0, x_off = 64, job_smem = 0;
    bool fused = false;      // activation quantization inside the GEMV kernel
    bool quant_ws = false;   // activation quantization by a separate kernel into ws
    Ring ring;
    size_t ws_xq = 0, ws_xd = 0, ws_xs = 0, ws_part = 0, ws_total = 0;
};

// have_xq: the caller passes quantized activations (qg_gemv_q).
inline GemvPlan plan_gemv(int fmt, int N, int K, int M, bool have_xq, int sms) {
    GemvPlan p;
    FmtInfo f;
    if (!fmt_info(fmt, f) || N < 1 || K < f.qk || K % f.qk || M < 1 || M > M_MAX || sms < 1) return p;
    p.nbr = K / f.qk;
    p.rb = (uint32_t)(p.nbr * f.bs);
    if (N < G_PLAN / 2) p.KS = std::min(p.nbr, (G_PLAN + N - 1) / N);
    p.groups = p.KS == 1 ? std::min(N, sms) : N;
    p.grid = p.groups * p.KS;
    p.MT = pick_mt(M);
    p.kslice_max = (p.nbr + p.KS - 1) / p.KS * f.qk;
    p.fused = !have_xq && xarea_bytes(M, p.kslice_max) + 64 <= XSMEM_CAP;
    p.quant_ws = !have_xq && !p.fused;
    p.job_smem = (uint32_t)align_up(64 + (p.fused ? xarea_bytes(M, p.kslice_max) : 0), 16);
    const uint32_t tb = stage_budget(p.job_smem);
    const int rows_per_cta = (N + p.groups - 1) / p.groups;
    uint32_t stage_bytes;
    if (p.KS == 1 && p.rb + 32 <= tb) {
        p.R = std::min<long>(std::min<long>(PART_SLOTS / p.MT, (tb - 32) / p.rb), rows_per_cta);
        p.segb = 0;
        stage_bytes = (uint32_t)p.R * p.rb;
    } else {
        p.R = 1;
        p.segb = std::max<int>(1, (int)((tb - 32) / (uint32_t)f.bs));
        const int slice_blocks = (p.nbr + p.KS - 1) / p.KS;
        stage_bytes = (uint32_t)(std::min(p.segb, slice_blocks) * f.bs);
    }
    p.ring = plan_ring(stage_bytes, p.job_smem);
    if (!p.ring.ok) return p;
    size_t o = 0;
    if (p.quant_ws) {
        p.ws_xq = o;
        o = align_up(o + (size_t)M * K, 256);
        p.ws_xd = o;
        o = align_up(o + 4ull * M * (K / 32), 256);
        p.ws_xs = o;
        o = align_up(o + 4ull * M * (K / 32), 256);
    }
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
    int nbr = 0, grid = 1, MT = 1, R = 0;
    uint32_t rb = 0, x_off = 0, job_smem = 0;
    bool fused = false;
    Ring ring;
    GemvPlan down;  // y = Wd h, h (fp32) in ws
    size_t ws_g = 0, ws_u = 0, ws_h = 0, ws_xq = 0, ws_xd = 0, ws_xs = 0, ws_down = 0, ws_total = 0;
};

inline FfnPlan plan_ffn(int fmt, int M, int H, int I, int sms) {
    FfnPlan p;
    FmtInfo f;
    if (!fmt_info(fmt, f) || M < 1 || M > M_MAX || H < f.qk || H % f.qk || I < f.qk || I % f.qk || sms < 1)
        return p;
    p.nbr = H / f.qk;
    p.rb = (uint32_t)(p.nbr * f.bs);
    p.MT = pick_mt(M);
    p.grid = std::min(I, sms);
    p.fused = xarea_bytes(M, H) <= XSMEM_CAP;
    p.job_smem = (uint32_t)align_up(p.fused ? xarea_bytes(M, H) : 16, 16);
    uint32_t tb = stage_budget(p.job_smem);
    if (2 * p.rb + 64 > tb) tb = (uint32_t)align_up(2 * p.rb + 64, 16);  // one pair per slot
    const int rows_per_cta = (I + p.grid - 1) / p.grid;
    p.R = (int)std::min<long>(std::min<long>(PART_SLOTS / (2 * p.MT), (tb - 64) / (2 * p.rb)), rows_per_cta);
    if (p.R < 1) return p;
    p.ring = plan_ring(2u * p.R * p.rb + 32, p.job_smem);
    if (!p.ring.ok) return p;
    p.down = plan_gemv(fmt, H, I, M, false, sms);
    if (!p.down.ok) return p;
    size_t o = 0;
    p.ws_g = o; o = align_up(o + 4ull * M * I, 256);
    p.ws_u = o; o = align_up(o + 4ull * M * I, 256);
    p.ws_h = o; o = align_up(o + 4ull * M * I, 256);
    if (!p.fused) {
        p.ws_xq = o; o = align_up(o + (size_t)M * H, 256);
        p.ws_xd = o; o = align_up(o + 4ull * M * (H / 32), 256);
        p.ws_xs = o; o = align_up(o + 4ull * M * (H / 32), 256);
    }
    p.ws_down = o;
    o = align_up(o + p.down.ws_total, 256);
    p.ws_total = o;
    p.ok = true;
    return p;
}

// ----------------------------------------------------------------------------- MoE FFN
struct MoePlan {
    bool ok = false;
    int S = 0, nbr_h = 0, nbr_i = 0;
    uint32_t rb_gu = 0, rb_d = 0;
    // router
    int router_grid = 0;
    // gate/up
    int gu_grid = 0, gu_R = 0;
    bool gu_fused = false;
    uint32_t gu_x_off = 0, gu_job = 0;
    Ring gu_ring;
    // down
    int dn_grid = 0, dn_R = 0, dn_nloc = 0;
    bool dn_fused = false;
    uint32_t dn_x_off = 0, dn_job = 0;
    Ring dn_ring;
    size_t ws_g = 0, ws_u = 0, ws_h = 0, ws_hq = 0, ws_hd = 0, ws_hs = 0, ws_logits = 0, ws_ids = 0, ws_w = 0,
           ws_xq = 0, ws_xd = 0, ws_xs = 0, ws_total = 0;
};

inline MoePlan plan_moe(int fmt, int M, int H, int E, int topk, int I, int sms) {
    MoePlan p;
    FmtInfo f;
    if (!fmt_info(fmt, f) || M < 1 || M > M_MAX || H < f.qk || H % f.qk || I < f.qk || I % f.qk || E < 1 ||
        E > 1024 || topk < 1 || topk > 16 || topk > E || sms < 1)
        return p;
    p.S = topk + 1;
    p.nbr_h = H / f.qk;
    p.nbr_i = I / f.qk;
    p.rb_gu = (uint32_t)(p.nbr_h * f.bs);
    p.rb_d = (uint32_t)(p.nbr_i * f.bs);
    p.router_grid = (E + 7) / 8;
    // gate/up
    const long pairs = (long)M * p.S * I;
    p.gu_grid = (int)std::min<long>(sms, pairs);
    p.gu_x_off = (uint32_t)align_up(4ull * M * topk, 16);
    p.gu_fused = p.gu_x_off + xarea_bytes(M, H) <= XSMEM_CAP;
    p.gu_job = (uint32_t)align_up(p.gu_x_off + (p.gu_fused ? xarea_bytes(M, H) : 0), 16);
    uint32_t tb = stage_budget(p.gu_job);
    if (2 * p.rb_gu + 64 > tb) tb = (uint32_t)align_up(2 * p.rb_gu + 64, 16);
    p.gu_R = (int)std::min<long>(PART_SLOTS / 2, (tb - 64) / (2 * p.rb_gu));
    if (p.gu_R < 1) return p;
    p.gu_ring = plan_ring(2u * p.gu_R * p.rb_gu + 32, p.gu_job);
    if (!p.gu_ring.ok) return p;
    // down
    p.dn_grid = std::min(sms, H);
    p.dn_nloc = (H + p.dn_grid - 1) / p.dn_grid;
    p.dn_x_off = (uint32_t)align_up(4ull * M * p.dn_nloc, 16);
    p.dn_fused = p.dn_x_off + xarea_bytes(M * p.S, I) <= XSMEM_CAP;
    p.dn_job = (uint32_t)align_up(p.dn_x_off + (p.dn_fused ? xarea_bytes(M * p.S, I) : 0), 16);
    uint32_t tbd = stage_budget(p.dn_job);
    if (p.rb_d + 32 > tbd) tbd = (uint32_t)align_up(p.rb_d + 32, 16);
    p.dn_R = (int)std::min<long>(std::min<long>(PART_SLOTS, (tbd - 32) / p.rb_d), p.dn_nloc);
    if (p.dn_R < 1) return p;
    p.dn_ring = plan_ring((uint32_t)p.dn_R * p.rb_d, p.dn_job);
    if (!p.dn_ring.ok) return p;
    // workspace
    const size_t R = (size_t)M * p.S;
    size_t o = 0;
    p.ws_g = o; o = align_up(o + 4 * R * I, 256);
    p.ws_u = o; o = align_up(o + 4 * R * I, 256);
    p.ws_h = o; o = align_up(o + 4 * R * I, 256);
    p.ws_hq = o; o = align_up(o + R * I, 256);
    p.ws_hd = o; o = align_up(o + 4 * R * (I / 32), 256);
    p.ws_hs = o; o = align_up(o + 4 * R * (I / 32), 256);
    p.ws_logits = o; o = align_up(o + 4ull * M * E, 256);
    p.ws_ids = o; o = align_up(o + 4ull * M * topk, 256);
    p.ws_w = o; o = align_up(o + 4ull * M * topk, 256);
    if (!p.gu_fused) {
        p.ws_xq = o; o = align_up(o + (size_t)M * H, 256);
        p.ws_xd = o; o = align_up(o + 4ull * M * (H / 32), 256);
        p.ws_xs = o; o = align_up(o + 4ull * M * (H / 32), 256);
    }
    p.ws_total = o;
    p.ok = true;
    return p;
}

}  // namespace qg
