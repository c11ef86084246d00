// qg_fmt.cu -- launchers of one block format.  The build compiles this file once per
// format with -DQG_FMT=<GGUF type id>, so the formats' kernels build in parallel.
#include <mutex>

#include "qg_jobs.cuh"
#include "qg_launch.h"

#ifndef QG_FMT
#error "QG_FMT must be defined"
#endif

namespace qg {

namespace {

// Opt-in to the full shared memory once per device and kernel instantiation.
template <class Kern>
bool allow_full_smem(Kern kern) {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

template <int FMT, int MT, class Job>
int launch_engine(const Job &job, int grid, uint32_t smem, cudaStream_t s) {
    auto kern = engine_kernel<FMT, MT, Job>;
    if (!allow_full_smem(kern)) return -4;
    kern<<<grid, NTHREADS, smem, s>>>(job);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

template <int FMT, class Job>
int launch_engine_mt(int MT, const Job &job, int grid, uint32_t smem, cudaStream_t s) {
    switch (MT) {
    case 1: return launch_engine<FMT, 1>(job, grid, smem, s);
    case 2: return launch_engine<FMT, 2>(job, grid, smem, s);
    case 4: return launch_engine<FMT, 4>(job, grid, smem, s);
    case 8: return launch_engine<FMT, 8>(job, grid, smem, s);
    case 16: return launch_engine<FMT, 16>(job, grid, smem, s);
    default: return -1;
    }
}

template <int FMT, bool XSM>
GemvJob<FMT, XSM> make_gemv_job(const GemvPlan &p, const GemvCall &c, const int8_t *xq, const float *xd,
                                const int32_t *xs, float *out) {
    GemvJob<FMT, XSM> j;
    j.nslots = p.ring.nslots;
    j.slot_bytes = p.ring.slot_bytes;
    j.job_smem_bytes = p.job_smem;
    j.W = c.W;
    j.Wend = c.W + (size_t)c.N * p.rb;
    j.N = c.N;
    j.K = c.K;
    j.M = c.M;
    j.nbr = p.nbr;
    j.KS = p.KS;
    j.groups = p.groups;
    j.R = p.R;
    j.segb = p.segb;
    j.rb = p.rb;
    j.x = c.x;
    j.xq = xq;
    j.xd = xd;
    j.xs = xs;
    j.out = out;
    j.slice_stride = (long)c.M * c.N;
    j.x_off = p.x_off;
    j.kslice_max = p.kslice_max;
    return j;
}

}  // namespace

template <int FMT>
int gemv_run_planned(const GemvPlan &p, const GemvCall &c) {
    if (p.ws_total && (c.ws == nullptr || c.ws_bytes < p.ws_total)) return -2;
    const int8_t *xq = c.xq;
    const float *xd = c.xd;
    const int32_t *xs = c.xs;
    if (p.quant_ws) {
        int8_t *q = reinterpret_cast<int8_t *>(c.ws + p.ws_xq);
        float *d = reinterpret_cast<float *>(c.ws + p.ws_xd);
        int32_t *s = reinterpret_cast<int32_t *>(c.ws + p.ws_xs);
        int rc = launch_quant_act(c.x, c.M, c.K, c.K, q, d, s, c.stream);
        if (rc) return rc;
        xq = q;
        xd = d;
        xs = s;
    }
    float *out = p.KS > 1 ? reinterpret_cast<float *>(c.ws + p.ws_part) : c.y;
    int rc;
    if (p.fused)
        rc = launch_engine_mt<FMT>(p.MT, make_gemv_job<FMT, true>(p, c, xq, xd, xs, out), p.grid,
                                   p.ring.smem_total, c.stream);
    else
        rc = launch_engine_mt<FMT>(p.MT, make_gemv_job<FMT, false>(p, c, xq, xd, xs, out), p.grid,
                                   p.ring.smem_total, c.stream);
    if (rc) return rc;
    if (p.KS > 1) return launch_splitk_reduce(out, p.KS, (long)c.M * c.N, c.y, c.stream);
    return 0;
}

template <int FMT>
int gemv_run(const GemvCall &c, int sms) {
    const GemvPlan p = plan_gemv(FMT, c.N, c.K, c.M, c.xq != nullptr, sms);
    if (!p.ok) return -1;
    return gemv_run_planned<FMT>(p, c);
}

template <int FMT>
int ffn_run(const FfnCall &c, int sms) {
    const FfnPlan p = plan_ffn(FMT, c.M, c.H, c.I, sms);
    if (!p.ok) return -1;
    if (c.ws == nullptr || c.ws_bytes < p.ws_total) return -2;
    float *g = reinterpret_cast<float *>(c.ws + p.ws_g);
    float *u = reinterpret_cast<float *>(c.ws + p.ws_u);
    float *h = reinterpret_cast<float *>(c.ws + p.ws_h);
    const int8_t *xq = nullptr;
    const float *xd = nullptr;
    const int32_t *xs = nullptr;
    if (!p.fused) {
        int8_t *q = reinterpret_cast<int8_t *>(c.ws + p.ws_xq);
        float *d = reinterpret_cast<float *>(c.ws + p.ws_xd);
        int32_t *s = reinterpret_cast<int32_t *>(c.ws + p.ws_xs);
        int rc = launch_quant_act(c.x, c.M, c.H, c.H, q, d, s, c.stream);
        if (rc) return rc;
        xq = q;
        xd = d;
        xs = s;
    }
    auto fill = [&](auto &j) {
        j.nslots = p.ring.nslots;
        j.slot_bytes = p.ring.slot_bytes;
        j.job_smem_bytes = p.job_smem;
        j.Wg = c.Wg;
        j.Wu = c.Wu;
        j.Wg_end = c.Wg + (size_t)c.I * p.rb;
        j.Wu_end = c.Wu + (size_t)c.I * p.rb;
        j.H = c.H;
        j.I = c.I;
        j.M = c.M;
        j.nbr = p.nbr;
        j.R = p.R;
        j.rb = p.rb;
        j.x = c.x;
        j.xq = xq;
        j.xd = xd;
        j.xs = xs;
        j.g_out = g;
        j.u_out = u;
        j.h_out = h;
        j.x_off = 0;
    };
    int rc;
    if (p.fused) {
        FfnGateUpJob<FMT, true> j;
        fill(j);
        rc = launch_engine_mt<FMT>(p.MT, j, p.grid, p.ring.smem_total, c.stream);
    } else {
        FfnGateUpJob<FMT, false> j;
        fill(j);
        rc = launch_engine_mt<FMT>(p.MT, j, p.grid, p.ring.smem_total, c.stream);
    }
    if (rc) return rc;
    GemvCall d{};
    d.W = c.Wd;
    d.N = c.H;
    d.K = c.I;
    d.M = c.M;
    d.x = h;
    d.y = c.y;
    d.ws = c.ws + p.ws_down;
    d.ws_bytes = c.ws_bytes - p.ws_down;
    d.stream = c.stream;
    return gemv_run_planned<FMT>(p.down, d);
}

template <int FMT>
int moe_run(const MoeCall &c, int sms) {
    const MoePlan p = plan_moe(FMT, c.M, c.H, c.E, c.topk, c.I, sms);
    if (!p.ok) return -1;
    if (c.ws == nullptr || c.ws_bytes < p.ws_total) return -2;
    using F = Fmt<FMT>;
    (void)sizeof(F);
    float *logits = reinterpret_cast<float *>(c.ws + p.ws_logits);
    int32_t *ids = reinterpret_cast<int32_t *>(c.ws + p.ws_ids);
    float *w = reinterpret_cast<float *>(c.ws + p.ws_w);
    float *g = reinterpret_cast<float *>(c.ws + p.ws_g);
    float *u = reinterpret_cast<float *>(c.ws + p.ws_u);
    float *h = reinterpret_cast<float *>(c.ws + p.ws_h);
    int8_t *hq = reinterpret_cast<int8_t *>(c.ws + p.ws_hq);
    float *hd = reinterpret_cast<float *>(c.ws + p.ws_hd);
    int32_t *hs = reinterpret_cast<int32_t *>(c.ws + p.ws_hs);

    int rc = launch_router_logits(c.x, c.M, c.H, c.Wr, c.E, logits, c.stream);
    if (rc) return rc;

    const int8_t *xq = nullptr;
    const float *xd = nullptr;
    const int32_t *xs = nullptr;
    if (!p.gu_fused) {
        int8_t *q = reinterpret_cast<int8_t *>(c.ws + p.ws_xq);
        float *d = reinterpret_cast<float *>(c.ws + p.ws_xd);
        int32_t *s = reinterpret_cast<int32_t *>(c.ws + p.ws_xs);
        rc = launch_quant_act(c.x, c.M, c.H, c.H, q, d, s, c.stream);
        if (rc) return rc;
        xq = q;
        xd = d;
        xs = s;
    }
    const size_t eb_gu = (size_t)c.I * p.rb_gu, eb_d = (size_t)c.H * p.rb_d;
    auto fill_gu = [&](auto &j) {
        j.nslots = p.gu_ring.nslots;
        j.slot_bytes = p.gu_ring.slot_bytes;
        j.job_smem_bytes = p.gu_job;
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
        j.H = c.H;
        j.I = c.I;
        j.M = c.M;
        j.nbr = p.nbr_h;
        j.R = p.gu_R;
        j.rb = p.rb_gu;
        j.ebytes = eb_gu;
        j.logits = logits;
        j.ids_ws = ids;
        j.w_ws = w;
        j.ids_out = c.ids_out;
        j.w_out = c.w_out;
        j.x = c.x;
        j.xq = xq;
        j.xd = xd;
        j.xs = xs;
        j.g_out = g;
        j.u_out = u;
        j.h_out = h;
        j.x_off = p.gu_x_off;
    };
    if (p.gu_fused) {
        MoeGateUpJob<FMT, true> j;
        fill_gu(j);
        rc = launch_engine<FMT, 1>(j, p.gu_grid, p.gu_ring.smem_total, c.stream);
    } else {
        MoeGateUpJob<FMT, false> j;
        fill_gu(j);
        rc = launch_engine<FMT, 1>(j, p.gu_grid, p.gu_ring.smem_total, c.stream);
    }
    if (rc) return rc;

    if (!p.dn_fused) {
        rc = launch_quant_act(h, c.M * p.S, c.I, c.I, hq, hd, hs, c.stream);
        if (rc) return rc;
    }
    auto fill_dn = [&](auto &j) {
        j.nslots = p.dn_ring.nslots;
        j.slot_bytes = p.dn_ring.slot_bytes;
        j.job_smem_bytes = p.dn_job;
        j.Wd_exps = c.Wd_exps;
        j.Wd_sh = c.Wd_sh;
        j.Wd_exps_end = c.Wd_exps + eb_d * c.E;
        j.Wd_sh_end = c.Wd_sh + eb_d;
        j.E = c.E;
        j.topk = c.topk;
        j.H = c.H;
        j.I = c.I;
        j.M = c.M;
        j.nbr = p.nbr_i;
        j.R = p.dn_R;
        j.nloc_max = p.dn_nloc;
        j.rb = p.rb_d;
        j.ebytes = eb_d;
        j.ids_ws = ids;
        j.w_ws = w;
        j.h = h;
        j.hq = hq;
        j.hd = hd;
        j.hs = hs;
        j.hq_ws = hq;
        j.hd_ws = hd;
        j.hs_ws = hs;
        j.y = c.y;
        j.x_off = p.dn_x_off;
    };
    if (p.dn_fused) {
        MoeDownJob<FMT, true> j;
        fill_dn(j);
        rc = launch_engine<FMT, 1>(j, p.dn_grid, p.dn_ring.smem_total, c.stream);
    } else {
        MoeDownJob<FMT, false> j;
        fill_dn(j);
        rc = launch_engine<FMT, 1>(j, p.dn_grid, p.dn_ring.smem_total, c.stream);
    }
    return rc;
}

// ----------------------------------------------------------------------------- test hook
// One thread per block: the block's bytes are copied into a private shared-memory window
// at the same offset modulo 16 as in global memory, then decoded with the GEMV decoders.
template <int FMT>
__global__ void __launch_bounds__(128) block_dots_kernel(const uint8_t *W, const int8_t *xq, const int32_t *xs,
                                                         int N, int K, int M, int32_t *dots, int32_t *aux) {
    using F = Fmt<FMT>;
    __shared__ __align__(16) uint8_t win[128 * 256];
    const int nbr = K / F::QK, nu = K / 32;
    const long g = (long)blockIdx.x * 128 + threadIdx.x;
    if (g >= (long)N * nbr) return;
    const int n = (int)(g / nbr), b = (int)(g % nbr);
    const uint8_t *src = W + g * F::BS;
    uint8_t *dst = win + threadIdx.x * 256 + ((uintptr_t)src & 15);
    for (int i = 0; i < F::BS; ++i) dst[i] = src[i];
    for (int j = 0; j < F::UPB; ++j) {
        WUnit w;
        F::decode(smem_addr(dst), j, w);
        const int u = b * F::UPB + j;
        for (int m = 0; m < M; ++m) {
            XUnit x;
            const int8_t *qa = xq + (size_t)m * K + 32 * (size_t)u;
            const uint4 a = ldg128_nc(qa), c = ldg128_nc(qa + 16);
            x.q[0] = a.x; x.q[1] = a.y; x.q[2] = a.z; x.q[3] = a.w;
            x.q[4] = c.x; x.q[5] = c.y; x.q[6] = c.z; x.q[7] = c.w;
            x.d = 0.0f;
            x.s = xs[(size_t)m * nu + u];
            const long o = ((long)m * N + n) * nu + u;
            dots[o] = F::idot(w, x);
            aux[o] = (FMT == F_Q4_K || FMT == F_Q5_K) ? x.s : 0;
        }
    }
}

template <int FMT>
int dots_run(const DotsCall &c) {
    using F = Fmt<FMT>;
    const long nblk = (long)c.N * (c.K / F::QK);
    const int grid = (int)((nblk + 127) / 128);
    block_dots_kernel<FMT><<<grid, 128, 0, c.stream>>>(c.W, c.xq, c.xs, c.N, c.K, c.M, c.dots, c.aux);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

template <int FMT>
int dev_err_take(unsigned int *err) {
    unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(err, g_qg_dev_err, sizeof(*err)) != cudaSuccess) return -4;
    if (cudaMemcpyToSymbol(g_qg_dev_err, &zero, sizeof(zero)) != cudaSuccess) return -4;
    return 0;
}

template int gemv_run<QG_FMT>(const GemvCall &, int);
template int gemv_run_planned<QG_FMT>(const GemvPlan &, const GemvCall &);
template int ffn_run<QG_FMT>(const FfnCall &, int);
template int moe_run<QG_FMT>(const MoeCall &, int);
template int dots_run<QG_FMT>(const DotsCall &);
template int dev_err_take<QG_FMT>(unsigned int *);

}  // namespace qg
