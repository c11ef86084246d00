// qg_fmt.cu -- launchers of one block format.  The build compiles this file once per
// format with -DQG_FMT=<GGUF type id>, so the formats' kernels build in parallel.
//
// Every operation is: a small preparation kernel that writes the activation tile image
// (normal launch), then an engine kernel launched with programmatic dependent launch, so
// that its weight streaming starts while the preparation is still running.
#include <mutex>
#include <type_traits>

#include "qg_jobs.cuh"
#include "qg_launch.h"
#include "qg_prefill.cuh"

#ifndef QG_FMT
#error "QG_FMT must be defined"
#endif

namespace qg {

namespace {

template <int V>
using ic = std::integral_constant<int, V>;

// Each kernel instantiation opts in to the full shared memory once per device; launches
// use programmatic stream serialization (see griddep_wait in qg_common.cuh).
template <int FMT, int T, int MT, int NCW, class Job, bool PAIR = false>
int launch_engine(const Job &job, int grid, uint32_t smem, cudaStream_t s) {
    static std::mutex mu;
    static bool ready[64] = {};
    auto kern = [] {
        if constexpr (PAIR)
            return engine_pair_kernel<FMT, T, MT, NCW, Job>;
        else
            return engine_kernel<FMT, T, MT, NCW, Job>;
    }();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -4;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX) != cudaSuccess ||
                cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                return -4;
            ready[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NCW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, job) != cudaSuccess) return -4;
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// The launch with MT tokens per lane and ncw warps (the default engine_ncw(), or NCW_WIDE
// where ncw_wide_allowed()).
template <int FMT, int T, int MT, class Job>
int launch_engine_ncw(int ncw, const Job &job, int grid, uint32_t smem, cudaStream_t s) {
    constexpr int TB = FT<FMT, T>::TASK_BYTES;
    if constexpr (ncw_wide_allowed(TB, MT)) {
        if (ncw == NCW_WIDE) return launch_engine<FMT, T, MT, NCW_WIDE>(job, grid, smem, s);
    }
    if (ncw != engine_ncw(TB, MT)) return -1;
    return launch_engine<FMT, T, MT, engine_ncw(TB, MT)>(job, grid, smem, s);
}

template <int FMT, int T, class Job>
int launch_engine_mt(int MT, int ncw, const Job &job, int grid, uint32_t smem, cudaStream_t s) {
    if constexpr (T == 16 || (T == 8 && (FMT == F_Q5_0 || FMT == F_Q8_0 || FMT == F_Q4_1 || FMT == F_Q5_1))) {
        // 16-block Q4_0 and 8-block Q4_1 / Q5_0 / Q5_1 / Q8_0 tasks are planned for one token
        // per lane only
        return MT == 1 ? launch_engine_ncw<FMT, T, 1>(ncw, job, grid, smem, s) : -1;
    }
    switch (MT) {
    case 1: return launch_engine_ncw<FMT, T, 1>(ncw, job, grid, smem, s);
    case 2: return launch_engine_ncw<FMT, T, 2>(ncw, job, grid, smem, s);
    case 4: return launch_engine_ncw<FMT, T, 4>(ncw, job, grid, smem, s);
    case 8: return launch_engine_ncw<FMT, T, 8>(ncw, job, grid, smem, s);
    case 16: return launch_engine_ncw<FMT, T, 16>(ncw, job, grid, smem, s);
    default: return -1;
    }
}

// The row-pair engine (engine_pair_kernel) for plain GEMV with two or more tokens: Q4_K,
// Q5_K, Q6_K and IQ4_XS one-superblock, Q4_0 / IQ4_NL 8-block and Q8_0 / Q4_1 / Q5_0 /
// Q5_1 4-block tasks of two rows, on 8 warps.
template <int FMT, int T, class Job>
int launch_pair(int MT, int ncw, const Job &job, int grid, uint32_t smem, cudaStream_t s) {
    if constexpr (((FMT == F_Q4_K || FMT == F_IQ4_XS) && T == 1) || ((FMT == F_Q4_0 || FMT == F_IQ4_NL) && T == 8) ||
                  ((FMT == F_Q8_0 || FMT == F_Q4_1 || FMT == F_Q5_0 || FMT == F_Q5_1) && T == 4) || FMT == F_Q5_K ||
                  FMT == F_Q6_K) {
        if (ncw != 8) return -1;
        switch (MT) {
        case 2: return launch_engine<FMT, T, 2, 8, Job, true>(job, grid, smem, s);
        case 4: return launch_engine<FMT, T, 4, 8, Job, true>(job, grid, smem, s);
        case 8: return launch_engine<FMT, T, 8, 8, Job, true>(job, grid, smem, s);
        case 16:
            if constexpr (FMT == F_Q5_K || FMT == F_Q6_K)
                return -1;  // not planned: see plan_gemv
            else
                return launch_engine<FMT, T, 16, 8, Job, true>(job, grid, smem, s);
        default: return -1;
        }
    } else {
        return -1;
    }
}

// Runs fn(ic<T>) with the task size the plan chose (see task_geo); LONG: the plan may have
// asked for long tasks.
template <bool LONG, class Fn>
int with_t(const TaskGeo &g, Fn &&fn) {
    if constexpr (QG_FMT == F_Q4_0 || QG_FMT == F_IQ4_NL) {
        if constexpr (LONG) {
            if (g.T == 16) return fn(ic<16>{});
        }
        if (g.T == 16) return -1;
        if (g.T == 8) return fn(ic<8>{});
        if (g.T == 4) return fn(ic<4>{});
        return fn(ic<1>{});
    } else if constexpr (QG_FMT == F_Q8_0 || QG_FMT == F_Q5_0 || QG_FMT == F_Q4_1 || QG_FMT == F_Q5_1) {
        if constexpr (LONG) {
            if (g.T == 8) return fn(ic<8>{});
        }
        if (g.T == 8) return -1;
        if (g.T == 4) return fn(ic<4>{});
        return fn(ic<1>{});
    } else if constexpr (QG_FMT == F_Q3_K || QG_FMT == F_Q5_K || QG_FMT == F_Q6_K) {
        return fn(ic<2>{});
    } else {
        if (g.T == 2) return fn(ic<2>{});
        return fn(ic<1>{});
    }
}

// The one-token engine (engine1_kernel) with ncw warps, for even task sizes (every stage one
// aligned bulk copy: see task_align_unit).
template <int FMT, int T>
int launch_engine1(int ncw, const Gemv1Args &a, int grid, uint32_t smem, cudaStream_t s) {
    if constexpr (FT<FMT, T>::TASK_BYTES % 2 != 0 || FT<FMT, T>::TPB != 1) {
        return -1;
    } else {
        static std::mutex mu;
        static bool ready[64][3] = {};
        const int v = ncw == 16 ? 2 : ncw == NCW_WIDE ? 1 : 0;
        auto kern = v == 2 ? engine1_kernel<FMT, T, 16> : v == 1 ? engine1_kernel<FMT, T, NCW_WIDE> : engine1_kernel<FMT, T, 8>;
        if (ncw != 16 && ncw != NCW_WIDE && ncw != 8) return -1;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -4;
        {
            std::lock_guard<std::mutex> lock(mu);
            if (!ready[dev][v]) {
                if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX) != cudaSuccess ||
                    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                    return -4;
                ready[dev][v] = true;
            }
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(ncw * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return -4;
        return cudaGetLastError() == cudaSuccess ? 0 : -4;
    }
}

// The FFN gate/up one-token kernel (ffn_gateup1_kernel) with ncw warps.
template <int FMT, int T>
int launch_ffn1(int ncw, const FfnGateUp1Args &a, int grid, uint32_t smem, cudaStream_t s) {
    if constexpr (FT<FMT, T>::TASK_BYTES % 2 != 0 || FT<FMT, T>::TPB != 1) {
        return -1;
    } else {
        static std::mutex mu;
        static bool ready[64][3] = {};
        const int v = ncw == 16 ? 2 : ncw == NCW_WIDE ? 1 : 0;
        auto kern = v == 2 ? ffn_gateup1_kernel<FMT, T, 16>
                           : v == 1 ? ffn_gateup1_kernel<FMT, T, NCW_WIDE> : ffn_gateup1_kernel<FMT, T, 8>;
        if (ncw != 16 && ncw != NCW_WIDE && ncw != 8) return -1;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -4;
        {
            std::lock_guard<std::mutex> lock(mu);
            if (!ready[dev][v]) {
                if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX) != cudaSuccess ||
                    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                    return -4;
                ready[dev][v] = true;
            }
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(ncw * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return -4;
        return cudaGetLastError() == cudaSuccess ? 0 : -4;
    }
}

template <class J>
void set_engine(J &j, const Ring &r, int tpr_x, int ntok) {
    j.depth = r.depth;
    j.slot_bytes = r.slot_bytes;
    j.x_bytes = r.x_bytes;
    j.j_bytes = r.j_bytes;
    j.tpr_x = tpr_x;
    j.tps = r.tps;
    j.ntok = ntok;
    j.xrep = 0;
}

}  // namespace

// A row-pair GEMV plan (p.pair) of N rows against an activation tile image that is already
// written (ximg, per-token pitch ximg_pitch, tiles of p.geo.XGT units): out = W x.
template <int FMT>
// The tokens go in chunks of p.MC (one launch each; every launch streams the weights).
// With p.KS > 1 every launch writes partial sums of its K-slices to part ([KS][M][N]),
// added into y by one reduction at the end.
int gemv_pair_run(const GemvPlan &p, const uint8_t *W, int N, int M, const uint8_t *ximg, size_t ximg_pitch,
                  float *y, float *part, cudaStream_t stream) {
    if (p.KS > 1 && part == nullptr) return -1;
    float *out = p.KS > 1 ? part : y;
    for (int m0 = 0; m0 < M; m0 += p.MC) {
        const int rc = with_t<false>(p.geo, [&](auto Tc) {
            constexpr int T = decltype(Tc)::value;
            GemvJob<FMT, T> j;
            set_engine(j, p.ring, p.tpr_x, std::min(p.MC, M - m0));
            j.W = W;
            j.Wend = W + (size_t)N * p.geo.rb;
            j.N = N;
            j.KS = p.KS;
            j.groups = p.groups;
            j.gpr = p.geo.gpr;
            j.rb = p.geo.rb;
            j.ximg = ximg + (size_t)m0 * ximg_pitch;
            j.ximg_pitch = (uint32_t)ximg_pitch;
            j.out = out + (size_t)m0 * N;
            j.slice_stride = (long)M * N;
            return launch_pair<FMT, T>(p.MT, p.ncw, j, p.grid, p.ring.smem_total, stream);
        });
        if (rc) return rc;
    }
    if (p.KS > 1) return launch_splitk_reduce(part, p.KS, (long)M * N, y, stream);
    return 0;
}

// A one-token plan (p.one) of N rows against an activation tile image that is already
// written: y = W x on engine1_kernel.
template <int FMT>
// ximg: the token's activation tile image, or nullptr with x: the fp32 row of K elements
// (device memory, 16-byte aligned), which every CTA quantizes itself.
int gemv_one_run(const GemvPlan &p, const uint8_t *W, int N, const uint8_t *ximg, const float *x, int K, float *y,
                 cudaStream_t stream) {
    return with_t<true>(p.geo, [&](auto Tc) {
        constexpr int T = decltype(Tc)::value;
        Gemv1Args a{};
        a.W = W;
        a.y = y;
        a.ximg = ximg;
        a.x = ximg ? nullptr : x;
        a.K = K;
        a.N = N;
        a.tpr = p.geo.tpr;
        a.depth = p.one_depth;
        a.xrep = p.xrep;
        a.ra = row_align_unit(p.geo.rb);
        a.nra = N / a.ra;
        a.rb = p.geo.rb;
        a.slot_bytes = p.one_slot;
        a.x_bytes = p.one_x;
        return launch_engine1<FMT, T>(p.ncw, a, p.grid, p.one_smem, stream);
    });
}

template <int FMT>
int gemv_run_planned(const GemvPlan &p, const GemvCall &c) {
    if (c.ws == nullptr || c.ws_bytes < p.ws_total) return -2;
    // one token of plain fp32 activations in device memory, rows of up to ONE_FUSED_K_MAX: the
    // one-token engine quantizes the row in every CTA, with no preparation kernel on the chain
    if (p.one && c.K <= ONE_FUSED_K_MAX && c.x && !c.u && !c.h_out && c.x_device && ((uintptr_t)c.x & 15u) == 0)
        return gemv_one_run<FMT>(p, c.W, c.N, nullptr, c.x, c.K, c.y, c.stream);
    uint8_t *ximg = c.ws + p.ws_ximg;
    int rc = launch_prep_tiles(c.x, c.u, c.h_out, c.xq, c.xd, c.xs, c.M, c.K, log2i(p.geo.XGT), ximg, nullptr,
                               nullptr, nullptr, c.stream);
    if (rc) return rc;
    if (p.pair)
        return gemv_pair_run<FMT>(p, c.W, c.N, c.M, ximg, p.ximg_pitch, c.y,
                                  p.KS > 1 ? reinterpret_cast<float *>(c.ws + p.ws_part) : nullptr, c.stream);
    if (p.one) return gemv_one_run<FMT>(p, c.W, c.N, ximg, nullptr, c.K, c.y, c.stream);
    float *out = p.KS > 1 ? reinterpret_cast<float *>(c.ws + p.ws_part) : c.y;
    rc = with_t<true>(p.geo, [&](auto Tc) {
        constexpr int T = decltype(Tc)::value;
        GemvJob<FMT, T> j;
        set_engine(j, p.ring, p.tpr_x, c.M);
        j.xrep = p.xrep;
        j.W = c.W;
        j.Wend = c.W + (size_t)c.N * p.geo.rb;
        j.N = c.N;
        j.KS = p.KS;
        j.groups = p.groups;
        j.gpr = p.geo.gpr;
        j.rb = p.geo.rb;
        j.ximg = ximg;
        j.ximg_pitch = (uint32_t)p.ximg_pitch;
        j.out = out;
        j.slice_stride = (long)c.M * c.N;
        return launch_engine_mt<FMT, T>(p.MT, p.ncw, j, p.grid, p.ring.smem_total, c.stream);
    });
    if (rc) return rc;
    if (p.KS > 1) return launch_splitk_reduce(out, p.KS, (long)c.M * c.N, c.y, c.stream);
    return 0;
}

template <int FMT>
int gemv_run(const GemvCall &c, int sms) {
    const GemvPlan p = plan_gemv(FMT, c.N, c.K, c.M, sms);
    if (!p.ok) return -1;
    return gemv_run_planned<FMT>(p, c);
}

template <int FMT>
int ffn_run(const FfnCall &c, int sms) {
    const FfnPlan p = plan_ffn(FMT, c.M, c.H, c.I, sms);
    if (!p.ok) return -1;
    if (c.ws == nullptr || c.ws_bytes < p.ws_total) return -2;
    uint8_t *ximg = c.ws + p.ws_ximg;
    float *g = reinterpret_cast<float *>(c.ws + p.ws_g);
    float *u = reinterpret_cast<float *>(c.ws + p.ws_u);
    float *h = reinterpret_cast<float *>(c.ws + p.ws_h);
    const int xgt = p.gate.pair ? p.gate.geo.XGT : p.geo.XGT;
    // one token in device memory with rows up to ONE_FUSED_K_MAX: the gate/up kernel quantizes x
    const bool fuse_x = p.one && c.H <= ONE_FUSED_K_MAX && c.x_device && ((uintptr_t)c.x & 15u) == 0;
    int rc = 0;
    if (!fuse_x) {
        rc = launch_prep_tiles(c.x, nullptr, nullptr, nullptr, nullptr, nullptr, c.M, c.H, log2i(xgt), ximg, nullptr,
                               nullptr, nullptr, c.stream);
        if (rc) return rc;
    }
    if (p.one) {
        // one token: gate/up with SwiGLU and the requantization of h in its epilogue, which
        // writes the down projection's tile image; then the down GEMV on it
        uint8_t *himg = c.ws + p.ws_down + p.down.ws_ximg;
        rc = with_t<true>(p.geo, [&](auto Tc) {
            constexpr int T = decltype(Tc)::value;
            FfnGateUp1Args a{};
            a.Wg = c.Wg;
            a.Wu = c.Wu;
            a.ximg = fuse_x ? nullptr : ximg;
            a.x = fuse_x ? c.x : nullptr;
            a.K = c.H;
            a.g_out = g;
            a.u_out = u;
            a.h_out = h;
            a.himg = himg;
            a.I = c.I;
            a.tpr = p.geo.tpr;
            a.depth = p.one_depth;
            a.xrep = XREP;
            a.himg_tpr = p.down.geo.tpr;
            a.himg_xgt_log2 = log2i(p.down.geo.XGT);
            a.rb = p.geo.rb;
            a.slot_bytes = p.one_slot;
            a.x_bytes = p.one_x;
            return launch_ffn1<FMT, T>(p.one_ncw, a, p.one_grid, p.one_smem, c.stream);
        });
        if (rc) return rc;
        return gemv_one_run<FMT>(p.down, c.Wd, c.H, himg, nullptr, c.I, c.y, c.stream);
    }
    if (p.gate.pair) {
        // several tokens: gate and up as two row-pair launches on the same tile image
        rc = gemv_pair_run<FMT>(p.gate, c.Wg, c.I, c.M, ximg, p.ximg_pitch, g, nullptr, c.stream);
        if (rc) return rc;
        rc = gemv_pair_run<FMT>(p.gate, c.Wu, c.I, c.M, ximg, p.ximg_pitch, u, nullptr, c.stream);
        if (rc) return rc;
    }
    for (int ch = 0; ch < (p.gate.pair ? 0 : p.nchunk); ++ch) {
        const int m0 = ch * p.MC, mc = std::min(p.MC, c.M - m0);
        rc = with_t<true>(p.geo, [&](auto Tc) {
            constexpr int T = decltype(Tc)::value;
            FfnGateUpJob<FMT, T> j;
            set_engine(j, p.ring, p.geo.tpr, mc);
            j.Wg = c.Wg;
            j.Wu = c.Wu;
            j.Wg_end = c.Wg + (size_t)c.I * p.geo.rb;
            j.Wu_end = c.Wu + (size_t)c.I * p.geo.rb;
            j.I = c.I;
            j.m0 = m0;
            j.rb = p.geo.rb;
            j.ximg = ximg;
            j.ximg_pitch = (uint32_t)p.ximg_pitch;
            j.g_out = g;
            j.u_out = u;
            return launch_engine_mt<FMT, T>(p.MT, p.ncw, j, p.grid, p.ring.smem_total, c.stream);
        });
        if (rc) return rc;
    }
    GemvCall d{};
    d.W = c.Wd;
    d.N = c.H;
    d.K = c.I;
    d.M = c.M;
    d.x = g;  // activations of the down projection: h = silu(g) * u
    d.u = u;
    d.h_out = h;
    d.y = c.y;
    d.ws = c.ws + p.ws_down;
    d.ws_bytes = c.ws_bytes - p.ws_down;
    d.stream = c.stream;
    return gemv_run_planned<FMT>(p.down, d);
}

// P activation rows per token: 1 (int8) or 2 (the two int8 planes of s16 activations).
template <int FMT, int P>
int moe_run_p(const MoeCall &c, const MoePlan &p) {
    float *logits = reinterpret_cast<float *>(c.ws + p.ws_logits);
    int32_t *ids = reinterpret_cast<int32_t *>(c.ws + p.ws_ids);
    float *w = reinterpret_cast<float *>(c.ws + p.ws_w);
    float *g = reinterpret_cast<float *>(c.ws + p.ws_g);
    float *u = reinterpret_cast<float *>(c.ws + p.ws_u);
    float *h = reinterpret_cast<float *>(c.ws + p.ws_h);
    int8_t *hq = reinterpret_cast<int8_t *>(c.ws + p.ws_hq);
    float *hd = reinterpret_cast<float *>(c.ws + p.ws_hd);
    int32_t *hs = reinterpret_cast<int32_t *>(c.ws + p.ws_hs);
    uint8_t *ximg = c.ws + p.ws_ximg, *himg = c.ws + p.ws_himg;

    int rc = launch_router_prep(c.x, c.M, c.H, c.Wr, c.E, logits, log2i(p.gh.XGT), ximg, P == 2, c.stream);
    if (rc) return rc;
    const size_t eb_gu = (size_t)c.I * p.gh.rb, eb_d = (size_t)c.H * p.gi.rb;
    rc = with_t<false>(p.gh, [&](auto Tc) {
        constexpr int T = decltype(Tc)::value;
        MoeGateUpJob<FMT, T, P> j;
        set_engine(j, p.gu_ring, p.gh.tpr, P);
        j.Wg_exps = c.Wg_exps;
        j.Wu_exps = c.Wu_exps;
        j.Wg_sh = c.Wg_sh;
        j.Wu_sh = c.Wu_sh;
        j.Wg_exps_end = c.Wg_exps + eb_gu * c.E;
        j.Wu_exps_end = c.Wu_exps + eb_gu * c.E;
        j.Wg_sh_end = c.Wg_sh + eb_gu;
        j.Wu_sh_end = c.Wu_sh + eb_gu;
        j.E = c.E;
        j.topk = c.topk;
        j.I = c.I;
        j.M = c.M;
        j.nunits = c.M * p.S * (c.I / 32);
        j.div_slots = FastDiv::make((uint32_t)p.S);
        j.div_ub = FastDiv::make((uint32_t)(c.I / 32));
        j.rb = p.gh.rb;
        j.ebytes = eb_gu;
        j.logits = logits;
        j.ids_ws = ids;
        j.w_ws = w;
        j.ids_out = c.ids_out;
        j.w_out = c.w_out;
        j.ximg = ximg;
        j.ximg_pitch = (uint32_t)p.ximg_pitch;
        j.g_out = g;
        j.u_out = u;
        // the epilogue writes h requantized (P image rows per token and slot) for the down
        // projection, and the plain h and its codes for callers
        j.himg = himg;
        j.himg_tpr = p.gi.tpr;
        j.himg_xgt_log2 = log2i(p.gi.XGT);
        j.h_out = h;
        j.hq = hq;
        j.hd = hd;
        j.hs = hs;
        return launch_engine_ncw<FMT, T, P>(p.gu_ncw, j, p.gu_grid, p.gu_ring.smem_total, c.stream);
    });
    if (rc) return rc;
    for (int ch = 0; ch < p.dn_nchunk; ++ch) {
        const int m0 = ch * p.dn_MC, mc = std::min(p.dn_MC, c.M - m0);
        rc = with_t<false>(p.gi, [&](auto Tc) {
            constexpr int T = decltype(Tc)::value;
            MoeDownJob<FMT, T, P> j;
            set_engine(j, p.dn_ring, p.gi.tpr, P);
            j.Wd_exps = c.Wd_exps;
            j.Wd_sh = c.Wd_sh;
            j.Wd_exps_end = c.Wd_exps + eb_d * c.E;
            j.Wd_sh_end = c.Wd_sh + eb_d;
            j.E = c.E;
            j.topk = c.topk;
            j.H = c.H;
            j.M = mc;
            j.m0 = m0;
            j.rb = p.gi.rb;
            j.ebytes = eb_d;
            j.ids_ws = ids;
            j.w_ws = w;
            j.ximg = himg;
            j.ximg_pitch = (uint32_t)p.himg_pitch;
            j.y = c.y;
            return launch_engine_ncw<FMT, T, P>(p.dn_ncw, j, p.dn_grid, p.dn_ring.smem_total, c.stream);
        });
        if (rc) return rc;
    }
    return 0;
}

template <int FMT>
int moe_run(const MoeCall &c, int sms) {
    const MoePlan p = plan_moe(FMT, c.M, c.H, c.E, c.topk, c.I, sms, c.s16);
    if (!p.ok) return -1;
    if (c.ws == nullptr || c.ws_bytes < p.ws_total) return -2;
    return c.s16 ? moe_run_p<FMT, 2>(c, p) : moe_run_p<FMT, 1>(c, p);
}

// ----------------------------------------------------------------------------- test hook
// Exact per-unit integer sums through the same format code as the GEMV (DotSink instead of
// the accumulating sink).  One thread per task: the task's block bytes are copied into a
// private shared-memory window at the same offset modulo 16 as in global memory, and the
// token's activation tile is built next to it.
struct DotSink {
    static constexpr int MT = 1;
    static constexpr bool DOTS = true;
    int32_t *dots, *aux;
    long base;  // index of unit 0 of this task for this token
    bool kquant;
    __device__ __forceinline__ void unit(int, int u, int dot, int xs) {
        dots[base + u] = dot;
        aux[base + u] = kquant ? xs : 0;
    }
};

constexpr int HOOK_THREADS = 32, HOOK_WIN = 320, HOOK_TILE = 800;

template <int FMT, int T>
__global__ void __launch_bounds__(HOOK_THREADS) block_dots_kernel(const uint8_t *W, const int8_t *xq,
                                                                  const int32_t *xs, int N, int K, int M,
                                                                  int32_t *dots, int32_t *aux) {
    using F = FT<FMT, T>;
    using TL = Tile<F::XGT>;
    static_assert(F::BPT * F::BS + 15 <= HOOK_WIN && TL::STRIDE <= HOOK_TILE, "test-hook window too small");
    __shared__ __align__(16) uint8_t mem[HOOK_THREADS * (HOOK_WIN + HOOK_TILE)];
    const int nbr = K / F::QK, nu = K / 32;
    const int tpr = nbr / F::BPT * F::TPB;
    const long task = (long)blockIdx.x * HOOK_THREADS + threadIdx.x;
    if (task >= (long)N * tpr) return;
    const int n = (int)(task / tpr), tt = (int)(task % tpr);
    const uint8_t *src = W + (size_t)n * nbr * F::BS + (size_t)(tt / F::TPB) * F::BPT * F::BS;
    uint8_t *win = mem + threadIdx.x * (HOOK_WIN + HOOK_TILE);
    uint8_t *blk = win + ((uintptr_t)src & 15);
    for (int i = 0; i < F::BPT * F::BS; ++i) blk[i] = src[i];
    uint8_t *tile = win + HOOK_WIN;
    for (int m = 0; m < M; ++m) {
        for (int u = 0; u < F::XGT; ++u) {
            const int xb = tt * F::XGT + u;
            int hs = 0, sum = 0;
            for (int i = 0; i < 32; ++i) {
                const int q = xq[(long)m * K + 32L * xb + i];
                tile[32 * u + i] = (uint8_t)q;
                sum += q;
                if (i < 16) hs += q;
            }
            reinterpret_cast<float *>(tile + TL::D)[u] = 0.0f;
            reinterpret_cast<int32_t *>(tile + TL::S)[u] = xs[(long)m * nu + xb];
            reinterpret_cast<uint32_t *>(tile + TL::H)[u] =
                ((uint32_t)hs & 0xffffu) | ((uint32_t)(sum - hs) << 16);
            reinterpret_cast<float *>(tile + TL::Q)[u] = 0.0f;
        }
        DotSink sink{dots, aux, ((long)m * N + n) * nu + (long)tt * F::XGT, FMT == F_Q4_K || FMT == F_Q5_K || FMT == F_Q4_1 || FMT == F_Q5_1 || FMT == F_Q2_K};
        F::run(blk, tt % F::TPB, XT{tile, 0}, 1, sink);
    }
}

template <int FMT>
int dots_run(const DotsCall &c) {
    const TaskGeo g = task_geo(FMT, c.K, c.M == 1);
    if (!g.ok) return -1;
    const long ntask = (long)c.N * g.tpr;
    const int grid = (int)((ntask + HOOK_THREADS - 1) / HOOK_THREADS);
    with_t<true>(g, [&](auto Tc) {
        constexpr int T = decltype(Tc)::value;
        block_dots_kernel<FMT, T><<<grid, HOOK_THREADS, 0, c.stream>>>(c.W, c.xq, c.xs, c.N, c.K, c.M, c.dots,
                                                                       c.aux);
        return 0;
    });
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

template <int FMT>
int dev_err_take(unsigned int *err) {
    unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(err, g_qg_dev_err, sizeof(*err)) != cudaSuccess) return -4;
    if (cudaMemcpyToSymbol(g_qg_dev_err, &zero, sizeof(zero)) != cudaSuccess) return -4;
    return 0;
}

// ----------------------------------------------------------------------------- prefill GEMM
// The fp16 activation image (normal launch), then the tensor-core GEMM (programmatic
// dependent launch: its set-up overlaps the image), then the split-K reduction if any.
template <int FMT>
int prefill_run(const PrefillCall &c, int sms) {
    const PrefillPlan p = plan_prefill(FMT, c.N, c.K, c.M, sms);
    if (!p.ok) return -1;
    if (c.ws == nullptr || c.ws_bytes < p.ws_total) return -2;
    uint8_t *ximg = c.ws + p.ws_ximg;
    int rc = launch_prefill_x16(c.x, c.M, c.K, p.BT, p.ntt, p.nkt, ximg, c.stream);
    if (rc) return rc;
    static std::mutex mu;
    static bool ready[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -4;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[dev]) {
            if (cudaFuncSetAttribute(prefill_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX) !=
                cudaSuccess)
                return -4;
            ready[dev] = true;
        }
    }
    PrefillArgs a{};
    a.W = c.W;
    a.rb = p.rb;
    a.N = c.N;
    a.K = c.K;
    a.M = c.M;
    a.BT = p.BT;
    a.NT = p.NT;
    a.ntt = p.ntt;
    a.nkt = p.nkt;
    a.ktps = p.ktps;
    a.stages = p.stages;
    a.tmem_cols = p.tmem_cols;
    a.idesc = p.idesc;
    a.ximg = ximg;
    a.out = p.KS > 1 ? reinterpret_cast<float *>(c.ws + p.ws_part) : c.y;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nn, (unsigned)p.ngrp, (unsigned)p.KS);
    cfg.blockDim = dim3(PF_THREADS);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, prefill_kernel<FMT>, a) != cudaSuccess) return -4;
    if (cudaGetLastError() != cudaSuccess) return -4;
    if (p.KS > 1) return launch_splitk_reduce(a.out, p.KS, (long)c.M * c.N, c.y, c.stream);
    return 0;
}

template <int FMT>
int dequant_f16_run(const uint8_t *W, int N, int K, uint16_t *out, cudaStream_t s) {
    FmtInfo f;
    if (!fmt_info(FMT, f)) return -1;
    const long total = (long)N * (K / 32);
    const int grid = (int)std::min<long>((total + 255) / 256, 8192);
    dequant_f16_kernel<FMT><<<grid, 256, 0, s>>>(W, (uint32_t)((K / f.qk) * f.bs), N, K, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

template int gemv_run<QG_FMT>(const GemvCall &, int);
template int gemv_run_planned<QG_FMT>(const GemvPlan &, const GemvCall &);
template int ffn_run<QG_FMT>(const FfnCall &, int);
template int moe_run<QG_FMT>(const MoeCall &, int);
template int dots_run<QG_FMT>(const DotsCall &);
template int dev_err_take<QG_FMT>(unsigned int *);
template int prefill_run<QG_FMT>(const PrefillCall &, int);
template int dequant_f16_run<QG_FMT>(const uint8_t *, int, int, uint16_t *, cudaStream_t);

}  // namespace qg
