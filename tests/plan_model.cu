// plan_model.cu -- a host model of the streaming engines' stage layout, checked against the
// planner for a sweep of shapes (GEMV, FFN sublayer, MoE FFN; every block format; 1..16
// tokens).  For every CTA, warp and stage of every planned launch it rebuilds, the way the
// kernels do, the runs of weight bytes a stage copies and the address every lane decodes,
// and checks: runs stay inside their tensor, the widened runs fit the ring slot, a run's
// tasks are adjacent in memory, every task is covered once, row-pair lanes find both rows'
// tasks, and no lane reads past its slot and its slack.  Test infrastructure: compiled and
// run by tests/test_plan_model.py on the CPU; prints "fails 0" when every check holds.
#include <cstdio>
#include <cstring>
#include <functional>
#include <vector>
#include "qg_plan.h"
using namespace qg;
static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { ++fails; if (fails < 20) { printf("FAIL %d: ", __LINE__); printf(__VA_ARGS__); printf("\n"); } } } while (0)
struct Cta { int o0, o1, tpr, grp, base = 0; };  // base: job-specific CTA origin (MoE gate/up: first unit)
static uint32_t toff(const TaskGeo &g, int tt) { return (uint32_t)((tt / g.TPB) * g.BPT * g.bs); }

void sim_c(const char *name, const TaskGeo &g, const Ring &r, int grid, int NCW, std::function<Cta(int)> cta,
           std::function<uintptr_t(const Cta &, int, int, uintptr_t &)> seg) {
    CHECK(r.ok, "%s ring not ok", name);
    CHECK(r.smem_total <= (uint32_t)SMEM_MAX, "%s smem %u", name, r.smem_total);
    for (int b = 0; b < grid; ++b) {
        Cta c = cta(b);
        const int ntask = (c.o1 - c.o0) * c.tpr, units = ntask / g.TPB;
        auto wstart = [&](int w) { return (int)((long)units * w / NCW) * g.TPB; };
        const int maxlen = (units + NCW - 1) / NCW * g.TPB, nchunk = (maxlen + r.tps - 1) / r.tps;
        for (int w = 0; w < NCW; ++w)
            for (int j = 0; j < nchunk; ++j) {
                const int fa = wstart(w) + j * r.tps, fb = std::min(wstart(w + 1), fa + r.tps);
                if (fa >= fb) continue;
                // pieces as the engine forms them: lane p takes group ga + p
                std::vector<std::pair<int, int>> pcs;
                if (c.grp == 0) pcs.push_back({fa, fb});
                else {
                    const int ga = (c.o0 + fa / c.tpr) / c.grp;
                    for (int p = 0; p < NPIECE_MAX; ++p) {
                        const long g0 = (long)(ga + p) * c.grp - c.o0;
                        const int ps = (int)std::max((long)fa, g0 * c.tpr), pe = (int)std::min((long)fb, (g0 + c.grp) * c.tpr);
                        if (ps < pe) pcs.push_back({ps, pe});
                    }
                    const long cend = ((long)(ga + NPIECE_MAX) * c.grp - c.o0) * c.tpr;
                    CHECK(cend >= fb, "%s b%d w%d j%d: stage needs more than %d pieces", name, b, w, j, NPIECE_MAX);
                }
                uint32_t off = 0;
                int covered = fa;
                for (auto &pc : pcs) {
                    CHECK(pc.first == covered, "%s gap in pieces", name);
                    CHECK((pc.second - pc.first) % g.TPB == 0, "%s piece not whole blocks", name);
                    const int o = pc.first / c.tpr, tt = pc.first - o * c.tpr;
                    uintptr_t lim;
                    const uintptr_t s0 = seg(c, c.o0 + o, tt, lim), e = s0 + toff(g, pc.second - pc.first);
                    CHECK(e <= lim, "%s piece past tensor end", name);
                    off += (uint32_t)(((e + 15) & ~(uintptr_t)15) - (s0 & ~(uintptr_t)15));
                    covered = pc.second;
                }
                CHECK(covered == fb, "%s stage not covered", name);
                CHECK(off <= r.slot_bytes, "%s slot overflow %u > %u", name, off, r.slot_bytes);
            }
    }
}

void sim(const char *name, const TaskGeo &g, const Ring &r, int grid, int NCW, std::function<Cta(int)> cta,
         std::function<uintptr_t(int, int, uintptr_t &)> seg) {
    sim_c(name, g, r, grid, NCW, cta, [&](const Cta &, int o, int tt, uintptr_t &lim) { return seg(o, tt, lim); });
}

// mirrors engine_pair_kernel: runs per stage, slot use, and every lane's two task addresses
// (whole rows: at most 3 runs that may span rows; K-slices: one run per row of each pair)
void sim_pair(const char *name, const GemvPlan &p, int N) {
    const TaskGeo &g = p.geo;
    const Ring &r = p.ring;
    CHECK(r.ok, "%s pair ring", name);
    const int P = (N + 1) / 2, NCW = p.ncw, KS = p.KS, ngroups = p.grid / KS;
    const bool split = KS > 1;
    CHECK(p.grid % KS == 0, "%s grid %d not a multiple of KS %d", name, p.grid, KS);
    const long TB = g.task_bytes();
    for (int cta = 0; cta < p.grid; ++cta) {
        const int grp = cta / KS, ks = cta % KS;
        const int t0 = (int)((long)g.gpr * ks / KS), tpr = (int)((long)g.gpr * (ks + 1) / KS) - t0;
        CHECK(tpr <= p.tpr_x, "%s slice of %d tasks past the tile area (%d)", name, tpr, p.tpr_x);
        if (split) CHECK(tpr >= PAIR_SPLIT_MIN_TPR, "%s slice of %d tasks", name, tpr);
        const int p0 = (int)((long)P * grp / ngroups), p1 = (int)((long)P * (grp + 1) / ngroups);
        const int ntask = (p1 - p0) * tpr;
        const int maxlen = (ntask + NCW - 1) / NCW, nchunk = (maxlen + r.tps - 1) / r.tps;
        for (int w = 0; w < NCW; ++w) {
            const int a = (int)((long)ntask * w / NCW), b = (int)((long)ntask * (w + 1) / NCW);
            for (int j = 0; j < nchunk; ++j) {
                const int fa = a + j * r.tps, fb = std::min(b, fa + r.tps);
                if (fa >= fb) continue;
                const int pa = fa / tpr, ca = fa - pa * tpr, pb = (fb - 1) / tpr, cb = fb - 1 - pb * tpr;
                const int ra = 2 * (p0 + pa), rz = 2 * (p0 + pb);
                const int nruns = split ? PAIR_RUNS_SPLIT : PAIR_RUNS;
                if (split) CHECK(pb - pa < PAIR_RUNS_SPLIT / 2, "%s stage over %d pairs", name, pb - pa + 1);
                long runrow[PAIR_RUNS_SPLIT], runcol[PAIR_RUNS_SPLIT], runn[PAIR_RUNS_SPLIT];
                bool valid[PAIR_RUNS_SPLIT];
                for (int k = 0; k < nruns; ++k) {
                    int row = 0, col = 0, n = 0;
                    if (split) {
                        const int pp = pa + k / 2;
                        if (pp <= pb) { row = 2 * (p0 + pp) + (k & 1); col = pp == pa ? ca : 0; n = (pp == pb ? cb + 1 : tpr) - col; }
                    } else if (k == 0) { row = ra; col = ca; n = pa == pb ? cb - ca + 1 : tpr - ca; }
                    else if (k == 1) { row = ra + 1; col = ca; n = pa == pb ? cb - ca + 1 : (tpr - ca) + (rz - ra - 2) * tpr + cb + 1; }
                    else if (pb > pa) { row = rz + 1; col = 0; n = cb + 1; }
                    valid[k] = n > 0 && row < N;
                    runrow[k] = row; runcol[k] = col; runn[k] = n;
                    if (valid[k]) {
                        if (split) CHECK(col + n <= tpr, "%s split run past its slice", name);
                        else CHECK((long)row * tpr + col + n <= (long)N * tpr, "%s run past end", name);
                    }
                }
                // slot offsets (the real byte addresses: slices start at t0 within the row)
                long off[PAIR_RUNS_SPLIT], tot = 0;
                for (int k = 0; k < nruns; ++k) {
                    off[k] = tot;
                    if (valid[k]) {
                        const long s0 = (long)runrow[k] * g.rb + (t0 + runcol[k]) * TB;
                        const long e = s0 + runn[k] * TB;
                        CHECK(e <= (long)N * g.rb, "%s run past the tensor", name);
                        tot += ((e + 15) & ~15L) - (s0 & ~15L);
                        off[k] += s0 & 15;
                    }
                }
                CHECK(tot <= (long)r.slot_bytes, "%s slot %ld > %u", name, tot, r.slot_bytes);
                // slot address of task (row, col): runs are row-major within the slice
                auto where = [&](long row, long col) -> long {
                    for (int k = 0; k < nruns; ++k) {
                        if (!valid[k]) continue;
                        if (split) {
                            if (row == runrow[k] && col >= runcol[k] && col < runcol[k] + runn[k]) return off[k] + (col - runcol[k]) * TB;
                            continue;
                        }
                        const long idx = (row * tpr + col) - (runrow[k] * tpr + runcol[k]);
                        if (idx >= 0 && idx < runn[k]) return off[k] + idx * TB;
                    }
                    return -1;
                };
                for (int l = 0; l < fb - fa; ++l) {
                    const int f = fa + l, pp = f / tpr, c = f - pp * tpr;
                    const int r0 = 2 * pp;  // CTA-relative
                    const long want0 = where(2L * (p0 + pp), c);
                    CHECK(want0 >= 0, "%s row0 not copied", name);
                    long got0, got1;
                    if (split) {
                        const int k = std::min(2 * (pp - pa), PAIR_RUNS_SPLIT - 2);
                        const long cofs = (long)(c - (pp == pa ? ca : 0)) * TB;
                        got0 = off[k] + cofs;
                        got1 = 2 * (p0 + pp) + 1 >= N ? got0 : off[k + 1] + cofs;
                    } else {
                        got0 = pp == pa ? off[0] + (long)(c - ca) * TB : off[1] + (long)((r0 - 2 * pa - 1) * tpr + c - ca) * TB;
                        got1 = 2 * (p0 + pp) + 1 >= N ? got0
                             : (pb > pa && pp == pb) ? off[2] + (long)c * TB : off[1] + (long)((r0 - 2 * pa) * tpr + c - ca) * TB;
                    }
                    CHECK(got0 == want0, "%s addr0 %ld != %ld (f %d pa %d pb %d)", name, got0, want0, f, pa, pb);
                    if (2 * (p0 + pp) + 1 < N) {
                        const long want1 = where(2L * (p0 + pp) + 1, c);
                        CHECK(want1 >= 0 && got1 == want1, "%s addr1 %ld != %ld", name, got1, want1);
                    }
                    CHECK(got0 + TB + 8 <= (long)r.slot_bytes + STAGE_SLACK && got1 + TB + 8 <= (long)r.slot_bytes + STAGE_SLACK,
                          "%s consumer read past slot", name);
                }
            }
        }
    }
}

int main() {
    const int sms = 152;
    const uintptr_t BASE = 0x7f0000000000ull;
    int fmts[] = {2, 3, 6, 7, 8, 10, 11, 12, 13, 14, 20, 23};
    int Ks[] = {32, 96, 256, 512, 544, 768, 1056, 2048, 4096, 5120, 17408, 7168, 14336, 2816};
    int Ns[] = {1, 2, 3, 5, 37, 64, 75, 76, 151, 152, 153, 300, 1024, 2048, 4096, 5120, 17408};
    int Ms[] = {1, 2, 3, 4, 5, 8, 16};
    int nplans = 0, npair = 0, none = 0, nffn1 = 0;
    char nm[160];
    for (int fmt : fmts) for (int K : Ks) for (int N : Ns) for (int M : Ms) {
        if (!task_geo(fmt, K, true).ok) continue;
        GemvPlan p = plan_gemv(fmt, N, K, M, sms);
        if (!p.ok) { CHECK(false, "gemv plan failed fmt %d N %d K %d M %d", fmt, N, K, M); continue; }
        ++nplans;
        const TaskGeo &g = p.geo;
        if (p.pair) {
            snprintf(nm, sizeof nm, "pair f%d N%d K%d M%d", fmt, N, K, M);
            // token chunks: MC tokens per launch, their tiles within the launch's x area
            CHECK(p.MC >= 1 && p.MC <= M && p.MC <= p.MT && p.MT >= 2, "%s chunk %d of %d (MT %d)", nm, p.MC, M, p.MT);

            CHECK((long)p.MC * p.tpr_x * g.stride <= (long)p.ring.x_bytes, "%s slice tiles", nm);
            if (p.KS > 1) CHECK(p.ws_part > 0 && p.ws_total >= p.ws_part + 4ull * p.KS * M * N, "%s partials", nm);
            sim_pair(nm, p, N);
            ++npair;
            continue;
        }
        if (p.one) {
            // one-token engine: per CTA, warp and stage a single bulk copy of whole tasks
            snprintf(nm, sizeof nm, "one f%d N%d K%d", fmt, N, K);
            ++none;
            const int ra = row_align_unit(g.rb), AU = task_align_unit(g.task_bytes());
            CHECK(M == 1 && p.KS == 1 && g.stage_aligned() && N % ra == 0 && 32 % AU == 0, "%s eligibility", nm);
            CHECK(p.one_smem <= (uint32_t)SMEM_MAX && p.one_depth >= 1, "%s smem %u", nm, p.one_smem);
            CHECK(p.one_x >= (uint32_t)((g.tpr + p.xrep) * g.stride) && p.xrep >= 31, "%s x tiles", nm);
            CHECK(p.one_slot == (uint32_t)(32 * g.task_bytes()), "%s slot", nm);
            const int TB = g.task_bytes(), S = p.ncw * p.one_depth;
            for (int b = 0; b < p.grid; ++b) {
                // CTA rows at multiples of ra, warp ranges at multiples of AU (engine1_kernel)
                const int o0 = ra * (int)((long)b * (N / ra) / p.grid), o1 = ra * (int)((long)(b + 1) * (N / ra) / p.grid);
                const int ntask = (o1 - o0) * g.tpr;
                CHECK(ntask % AU == 0, "%s CTA tasks %d not a multiple of %d", nm, ntask, AU);
                CHECK(engine1_smem(S, p.one_slot, p.one_x, ntask) <= p.one_smem, "%s part of CTA %d", nm, b);
                for (int w = 0; w < p.ncw; ++w) {
                    const int wa = AU * (int)((long)(ntask / AU) * w / p.ncw);
                    const int wb = AU * (int)((long)(ntask / AU) * (w + 1) / p.ncw);
                    for (int fa = wa; fa < wb; fa += 32) {
                        const int fb = std::min(wb, fa + 32);
                        const uintptr_t src = BASE + (uintptr_t)o0 * g.rb + (uintptr_t)fa * TB;
                        const uintptr_t end = src + (uintptr_t)(fb - fa) * TB;
                        CHECK(src % 16 == 0 && (end - src) % 16 == 0, "%s copy alignment", nm);
                        CHECK(end <= BASE + (uintptr_t)N * g.rb && src >= BASE, "%s copy range", nm);
                        CHECK((uint32_t)((fb - fa) * TB) <= p.one_slot, "%s slot overflow", nm);
                        for (int f = fa; f < fb; ++f) {
                            const int o = f / g.tpr, tt = f % g.tpr;
                            CHECK(o0 + o < o1, "%s row", nm);
                            // the task's bytes: row o, task tt
                            CHECK(BASE + (uintptr_t)(o0 + o) * g.rb + (uintptr_t)tt * TB == src + (uintptr_t)(f - fa) * TB,
                                  "%s contiguity", nm);
                            const int xc = fa % g.tpr + (f - fa);
                            CHECK(xc < g.tpr + p.xrep && xc % g.tpr == tt, "%s virtual column %d", nm, xc);
                            CHECK(f < ntask, "%s part index", nm);
                        }
                    }
                }
            }
            continue;
        }
        snprintf(nm, sizeof nm, "gemv f%d N%d K%d M%d KS%d", fmt, N, K, M, p.KS);
        CHECK(p.ring.x_bytes >= (uint32_t)(M * (p.tpr_x + p.xrep) * g.stride), "%s x bytes", nm);
        // repeated tiles: a stage's last lane reads virtual column (tpr - 1) + 31 at most
        CHECK(p.xrep == 0 || (p.xrep >= 31 && M == 1), "%s xrep %d", nm, p.xrep);
        const int KS = p.KS, groups = p.groups, gpr = g.gpr, TPB = g.TPB;
        sim(nm, g, p.ring, p.grid, p.ncw,
            [&](int b) { const int gg = b / KS, ks = b % KS; Cta c; c.o0 = (int)((long)gg * N / groups);
                         c.o1 = (int)((long)(gg + 1) * N / groups); const int t0 = (int)((long)ks * gpr / KS) * TPB;
                         c.tpr = (int)((long)(ks + 1) * gpr / KS) * TPB - t0; c.grp = KS == 1 ? 0 : 1;
                         CHECK(c.tpr <= p.tpr_x, "slice tpr"); return c; },
            [&](int o, int tt, uintptr_t &lim) { lim = BASE + (uintptr_t)N * g.rb; return BASE + (uintptr_t)o * g.rb + toff(g, tt); });
    }
    printf("gemv plans %d (row pairs %d, one-token %d)\n", nplans, npair, none);
    int Hs[] = {512, 1024, 2048, 4096, 5120, 7168}, Is[] = {256, 512, 1536, 2048, 14336, 17408};
    for (int fmt : fmts) for (int H : Hs) for (int I : Is) for (int M : Ms) {
        if (!task_geo(fmt, H, false).ok || !task_geo(fmt, I, false).ok) continue;
        FfnPlan p = plan_ffn(fmt, M, H, I, sms);
        if (!p.ok) { CHECK(false, "ffn plan failed fmt %d H %d I %d M %d", fmt, H, I, M); continue; }
        snprintf(nm, sizeof nm, "ffn f%d H%d I%d M%d", fmt, H, I, M);
        if (p.gate.pair) {
            CHECK(p.ximg_pitch >= (size_t)p.gate.tpr_x * p.gate.geo.stride, "%s gate pitch", nm);
            sim_pair(nm, p.gate, I);
            ++npair;
        }
        const TaskGeo &g = p.geo;
        if (p.one) {
            // one-token gate/up with the SwiGLU epilogue: units of 32 rows per CTA, the gate
            // rows then the up rows as two contiguous ranges; a stage at most two copies
            ++nffn1;
            const int AU = task_align_unit(g.task_bytes());
            CHECK(M == 1 && p.down.one && g.stage_aligned(), "%s one eligibility", nm);
            CHECK(p.one_smem <= (uint32_t)SMEM_MAX && p.one_depth >= 1, "%s one smem", nm);
            CHECK(p.one_x >= (uint32_t)((g.tpr + XREP) * g.stride), "%s one x tiles", nm);
            const int U = I / 32, TB = g.task_bytes(), S = p.one_ncw * p.one_depth;
            for (int b = 0; b < p.one_grid; ++b) {
                const int u0 = (int)((long)U * b / p.one_grid), u1 = (int)((long)U * (b + 1) / p.one_grid);
                const int nu = u1 - u0, G = 32 * nu * g.tpr, ntask = 2 * G;
                CHECK(G % AU == 0, "%s gate tasks %d not a multiple of %d", nm, G, AU);
                CHECK(engine1_smem(S, p.one_slot, p.one_x, ffn1_part_floats(nu, g.tpr)) <= p.one_smem, "%s part %d", nm, b);
                for (int w = 0; w < p.one_ncw; ++w) {
                    const int wa = AU * (int)((long)(ntask / AU) * w / p.one_ncw);
                    const int wb = AU * (int)((long)(ntask / AU) * (w + 1) / p.one_ncw);
                    for (int fa = wa; fa < wb; fa += 32) {
                        const int fb = std::min(wb, fa + 32), g1 = std::min(fb, G), ua = std::max(fa, G);
                        long bytes = 0;
                        if (fa < g1) {
                            const long off = (long)32 * u0 * g.rb + (long)fa * TB, n = (long)(g1 - fa) * TB;
                            CHECK(off % 16 == 0 && n % 16 == 0 && off + n <= (long)I * g.rb, "%s gate copy", nm);
                            bytes += n;
                        }
                        if (ua < fb) {
                            const long off = (long)32 * u0 * g.rb + (long)(ua - G) * TB, n = (long)(fb - ua) * TB;
                            CHECK(off % 16 == 0 && n % 16 == 0 && off + n <= (long)I * g.rb, "%s up copy", nm);
                            bytes += n;
                        }
                        CHECK(bytes == (long)(fb - fa) * TB && bytes <= (long)p.one_slot, "%s slot", nm);
                        for (int f = fa; f < fb; ++f) {
                            const int ff = f < G ? f : f - G, o = ff / g.tpr;
                            CHECK(o < 32 * nu && f < ntask, "%s task row", nm);
                            const int xc = fa % g.tpr + (f - fa);
                            CHECK(xc < g.tpr + XREP && xc % g.tpr == f % g.tpr && f % g.tpr == ff % g.tpr, "%s column", nm);
                        }
                    }
                }
                // h units into the down projection's tile image: tile (u >> xgt_log2) of one row
                CHECK((u1 - 1) / p.down.geo.XGT < p.down.geo.tpr, "%s h tile", nm);
            }
            CHECK(p.down.ximg_pitch >= (size_t)p.down.geo.tpr * p.down.geo.stride, "%s h image", nm);
        }
        sim(nm, g, p.ring, p.grid, p.ncw,
            [&](int b) { Cta c; c.o0 = (int)((long)b * 2 * I / p.grid); c.o1 = (int)((long)(b + 1) * 2 * I / p.grid);
                         c.tpr = g.tpr; c.grp = I; return c; },
            [&](int o, int tt, uintptr_t &lim) { const bool up = o >= I; const uintptr_t base = up ? BASE + (1ull << 36) : BASE;
                                                 lim = base + (uintptr_t)I * g.rb; return base + (uintptr_t)(up ? o - I : o) * g.rb + toff(g, tt); });
    }
    int Es[] = {16, 64, 256}, topks[] = {1, 4, 8}, mH[] = {512, 2048, 4096, 7168}, mI[] = {256, 512, 768, 1536};
    for (int fmt : fmts) for (int E : Es) for (int topk : topks) for (int H : mH) for (int I : mI) for (int M : Ms) {
        if (topk > E || !task_geo(fmt, H, false).ok || !task_geo(fmt, I, false).ok) continue;
      for (int P = 1; P <= 2; ++P) {
        MoePlan p = plan_moe(fmt, M, H, E, topk, I, sms, P == 2);
        if (!p.ok) {
            if ((long)M * P * task_geo(fmt, H, false).tpr * task_geo(fmt, H, false).stride <= (long)XCAP)
                CHECK(false, "moe plan failed f%d E%d k%d H%d I%d M%d P%d", fmt, E, topk, H, I, M, P);
            continue;
        }
        const int S = p.S;
        CHECK(p.P == P, "moe planes");
        snprintf(nm, sizeof nm, "moe-gu f%d E%d k%d H%d I%d M%d P%d", fmt, E, topk, H, I, M, P);
        const size_t eb = (size_t)I * p.gh.rb;
        const long units = (long)M * S * (I / 32);
        // units of 32 positions: CTA-local rows 64 * unit + 32 * up + (j & 31)
        sim_c(nm, p.gh, p.gu_ring, p.gu_grid, p.gu_ncw,
            [&](int b) { const int u0 = (int)(units * b / p.gu_grid), u1 = (int)(units * (b + 1) / p.gu_grid); Cta c;
                         c.o0 = 0; c.o1 = 64 * (u1 - u0); c.tpr = p.gh.tpr; c.grp = 32; c.base = u0;
                         CHECK((uint32_t)(4 * c.o1 * P) <= p.gu_ring.j_bytes, "moe gu jarea");
                         CHECK((uint32_t)(M * P * p.gh.tpr * p.gh.stride) <= p.gu_ring.x_bytes, "moe gu x"); return c; },
            [&](const Cta &c, int o, int tt, uintptr_t &lim) {
                const int un = c.base + (o >> 6), up = (o >> 5) & 1, gs = un / (I / 32), jj = 32 * (un % (I / 32)) + (o & 31);
                const int s = gs % S;
                uintptr_t base; if (s < topk) { base = (up ? BASE + (1ull << 38) : BASE) + (uintptr_t)((s * 37 + 5) % E) * eb; lim = (up ? BASE + (1ull << 38) : BASE) + eb * E; }
                else { base = up ? BASE + (3ull << 38) : BASE + (2ull << 38); lim = base + eb; }
                return base + (uintptr_t)jj * p.gh.rb + toff(p.gh, tt); });
        snprintf(nm, sizeof nm, "moe-dn f%d E%d k%d H%d I%d M%d P%d", fmt, E, topk, H, I, M, P);
        for (int ch = 0; ch < p.dn_nchunk; ++ch) {
            const int mc = std::min(p.dn_MC, M - ch * p.dn_MC);
            sim(nm, p.gi, p.dn_ring, p.dn_grid, p.dn_ncw,
                [&](int b) { const int n0 = (int)((long)b * H / p.dn_grid), n1 = (int)((long)(b + 1) * H / p.dn_grid); Cta c;
                             c.o0 = 0; c.o1 = mc * S * (n1 - n0); c.tpr = p.gi.tpr; c.grp = n1 - n0;
                             CHECK((uint32_t)(4 * c.o1 * P) <= p.dn_ring.j_bytes, "moe dn jarea");
                             CHECK((uint32_t)(mc * S * P * p.gi.tpr * p.gi.stride) <= p.dn_ring.x_bytes, "moe dn x"); return c; },
                [&](int o, int tt, uintptr_t &lim) { lim = BASE + (uintptr_t)H * p.gi.rb * (E + 1) * 32; return BASE + (uintptr_t)o * p.gi.rb + toff(p.gi, tt); });
        }
      }
    }
    // the launch shapes chosen for the decode FFN of hidden 5120 / inter 17408 (measured
    // choices; a change here changes the timings the documentation reports)
    {
        const GemvPlan a = plan_gemv(12, 17408, 5120, 1, sms), b = plan_gemv(12, 5120, 17408, 1, sms);
        CHECK(!a.pair && a.KS == 1 && a.ncw == 12 && a.xrep == XREP && a.geo.T == 2, "Q4_K 17408x5120 M1 plan");
        CHECK(!b.pair && b.KS == 1 && b.ncw == 12 && b.xrep == XREP, "Q4_K 5120x17408 M1 plan");
        const GemvPlan c = plan_gemv(2, 17408, 5120, 1, sms);
        CHECK(!c.pair && c.geo.T == 16 && c.xrep == XREP, "Q4_0 17408x5120 M1 plan");
        const GemvPlan d = plan_gemv(12, 17408, 5120, 4, sms);
        CHECK(d.pair && d.KS == 1 && d.MT == 4 && d.MC == 4, "Q4_K 17408x5120 M4 plan");
        const GemvPlan e = plan_gemv(12, 5120, 17408, 16, sms), f = plan_gemv(12, 5120, 17408, 8, sms);
        CHECK(e.pair && e.KS == 4 && e.MT == 16 && e.MC == 16 && e.grid == 152, "Q4_K 5120x17408 M16 plan: K-sliced pairs");
        CHECK(f.pair && f.KS == 2 && f.MT == 8, "Q4_K 5120x17408 M8 plan");
        const GemvPlan g6 = plan_gemv(14, 17408, 5120, 16, sms);
        CHECK(g6.pair && g6.MT == 8 && g6.MC == 8, "Q6_K 17408x5120 M16 plan: two launches of 8");
        const FfnPlan h = plan_ffn(12, 16, 5120, 17408, sms);
        CHECK(h.ok && h.gate.pair && h.gate.KS == 1 && h.down.pair && h.down.KS == 4, "FFN Q4_K M16 plan");
        const MoePlan m1 = plan_moe(12, 1, 2048, 256, 8, 512, sms), m2 = plan_moe(12, 1, 2048, 256, 8, 512, sms, true);
        CHECK(m1.ok && m1.P == 1 && m1.gu_grid == 144 && m2.ok && m2.P == 2, "MoE plans");
    }
    printf("one-token FFN plans %d\nfails %d\n", nffn1, fails);
    return fails != 0;
}
