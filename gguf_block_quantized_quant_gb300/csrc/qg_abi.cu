// qg_abi.cu -- the extern "C" boundary of libqg (declared in include/qg.h) and the
// format-independent kernels: activation quantization, split-K reduction, router logits.
//
// The boundary follows "01 · 阶段总览：从 2B 到 8B 再到 MoE", section 一: a pure C ABI module
// whose device call reports one status (0 = done on the GPU).  The page's host-side
// mapping of a failure to "the caller runs the CPU path" is deliberately not reproduced:
// a failure is returned as a negative status and nothing runs elsewhere.
#include <cuda.h>

#include <mutex>
#include <set>
#include <utility>

#include "../../include/qg.h"
#include "qg_jobs.cuh"
#include "qg_launch.h"

namespace qg {

// ----------------------------------------------------------------------------- kernels
// One warp per 32-element block (see quant_block_warp).
__global__ void __launch_bounds__(256) quant_act_kernel(const float *x, int M, int K, long ldx, int8_t *xq,
                                                        float *xd, int32_t *xs) {
    const int lane = threadIdx.x & 31;
    const int nb = K / 32;
    const long total = (long)M * nb;
    const long wpg = (long)gridDim.x * (blockDim.x >> 5);
    for (long w = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += wpg) {
        const int m = (int)(w / nb), b = (int)(w % nb);
        const float v = x[(long)m * ldx + 32 * b + lane];
        int q, s;
        float d;
        quant_block_warp(v, q, d, s);
        xq[(long)m * K + 32 * b + lane] = (int8_t)q;
        if (lane == 0) {
            xd[(long)m * nb + b] = d;
            xs[(long)m * nb + b] = s;
        }
    }
}

// s16 activation quantization in the plain layout (qg_quantize_act_s16).
__global__ void __launch_bounds__(256) quant_act_s16_kernel(const float *x, int M, int K, int16_t *xq, float *xd,
                                                            int32_t *xs) {
    const int lane = threadIdx.x & 31;
    const int nb = K / 32;
    const long total = (long)M * nb;
    const long wpg = (long)gridDim.x * (blockDim.x >> 5);
    for (long w = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += wpg) {
        const int m = (int)(w / nb), b = (int)(w % nb);
        int q, s;
        float d;
        quant_block_warp16(x[(long)m * K + 32 * b + lane], q, d, s);
        xq[(long)m * K + 32 * b + lane] = (int16_t)q;
        if (lane == 0) {
            xd[(long)m * nb + b] = d;
            xs[(long)m * nb + b] = s;
        }
    }
}

// y[i] = sum over the K-slices in slice order.
__global__ void splitk_reduce_kernel(const float *part, int KS, long MN, float *y) {
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < MN; i += (long)gridDim.x * blockDim.x) {
        float s = 0.0f;
        for (int k = 0; k < KS; ++k) s += part[(long)k * MN + i];
        y[i] = s;
    }
}

// Activation tile image (see prep_tiles_warp).  Launched as a programmatic dependent of the
// previous kernel in the stream: it lets its own dependent (the engine) start at once, then
// waits for the previous kernel to finish before it reads any input or writes the
// workspace.
__global__ void __launch_bounds__(256) prep_tiles_kernel(const float *x, const float *u, float *h_out,
                                                         const int8_t *xq, const float *xd, const int32_t *xs,
                                                         int rows, int K, int xgt_log2, uint8_t *img, int8_t *mq,
                                                         float *md, int32_t *ms) {
    griddep_launch_dependents();
    griddep_wait();
    const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
    const long wid = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    prep_tiles_warp(x, u, h_out, xq, xd, xs, rows, K, xgt_log2, img, mq, md, ms, wid, nwarps);
}

// Blocks [0, ceil(E/2)): logits[m][e] = sum_k Wr[e][k] * x[m][k] in fp32.  Each block takes
// two experts, four warps per expert, each warp a quarter of the row with 16-byte loads so
// that a lane's loads are all in flight at once; the quarters are added in order.  The
// remaining blocks write the activation tile image of x (int8 rows, or with s16 == true
// the two int8 planes of each s16 row).  Launched like prep_tiles_kernel.
constexpr int ROUTER_SPLIT = 4;  // warps per expert row
__global__ void __launch_bounds__(256) router_prep_kernel(const float *x, int M, int H, const float *Wr, int E,
                                                          float *logits, int xgt_log2, uint8_t *img, bool s16) {
    griddep_launch_dependents();
    griddep_wait();
    __shared__ float part[8][M_MAX];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int epb = 8 / ROUTER_SPLIT;  // experts per block
    const int nrouter = (E + epb - 1) / epb;
    if ((int)blockIdx.x >= nrouter) {
        const long nwarps = (long)(gridDim.x - nrouter) * (blockDim.x >> 5);
        const long wid = (long)(blockIdx.x - nrouter) * (blockDim.x >> 5) + warp;
        if (s16)
            prep_tiles_s16_warp(x, M, H, xgt_log2, img, wid, nwarps);
        else
            prep_tiles_warp(x, nullptr, nullptr, nullptr, nullptr, nullptr, M, H, xgt_log2, img, nullptr, nullptr,
                            nullptr, wid, nwarps);
        return;
    }
    const int e = blockIdx.x * epb + warp / ROUTER_SPLIT, q = warp % ROUTER_SPLIT;
    float acc[M_MAX];
#pragma unroll
    for (int m = 0; m < M_MAX; ++m) acc[m] = 0.0f;
    if (e < E) {
        const float *wr = Wr + (long)e * H;
        const int k0 = (int)((long)q * H / ROUTER_SPLIT), k1 = (int)((long)(q + 1) * H / ROUTER_SPLIT);
        if ((((uintptr_t)wr | (uintptr_t)x) & 15u) == 0 && ((k0 | k1) & 3) == 0) {
            const float4 *w4 = reinterpret_cast<const float4 *>(wr);
            // RCH 16-byte loads of the row per lane in flight at once, then, token by
            // token, the same number of loads of x (from L2: the previous kernel may have
            // written it); the products are added in k order
            constexpr int RCH = 4;
            for (int kb = (k0 >> 2) + lane; kb < (k1 >> 2); kb += 32 * RCH) {
                float4 wv[RCH];
#pragma unroll
                for (int i = 0; i < RCH; ++i)
                    wv[i] = kb + 32 * i < (k1 >> 2) ? __ldg(w4 + kb + 32 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int m = 0; m < M_MAX; ++m) {
                    if (m < M) {
                        const float4 *x4 = reinterpret_cast<const float4 *>(x + (long)m * H);
                        float4 xv[RCH];
#pragma unroll
                        for (int i = 0; i < RCH; ++i)
                            xv[i] = kb + 32 * i < (k1 >> 2) ? __ldcg(x4 + kb + 32 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < RCH; ++i) {
                            if (kb + 32 * i < (k1 >> 2)) {
                                acc[m] = fmaf(wv[i].x, xv[i].x, acc[m]);
                                acc[m] = fmaf(wv[i].y, xv[i].y, acc[m]);
                                acc[m] = fmaf(wv[i].z, xv[i].z, acc[m]);
                                acc[m] = fmaf(wv[i].w, xv[i].w, acc[m]);
                            }
                        }
                    }
                }
            }
        } else {
            for (int k = k0 + lane; k < k1; k += 32) {
                const float wv = __ldg(wr + k);
#pragma unroll
                for (int m = 0; m < M_MAX; ++m)
                    if (m < M) acc[m] = fmaf(wv, __ldcg(x + (long)m * H + k), acc[m]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < M_MAX; ++m) {
        if (m < M) {
            const float v = warp_sum(acc[m]);
            if (lane == 0) part[warp][m] = v;
        }
    }
    __syncthreads();
    if (e < E && q == 0 && lane < M) {
        float v = part[warp][lane];
        for (int r = 1; r < ROUTER_SPLIT; ++r) v += part[warp + r][lane];
        logits[(long)lane * E + e] = v;
    }
}

// fp16 activation image of the prefill GEMM (see launch_prefill_x16): one thread per 16-byte
// chunk of the image, in image order (coalesced stores).  Tiles are ordered K tile major,
// token tile minor; chunk position p of row r of a tile holds the 8 elements of logical chunk
// p ^ (r & 7) (the 128-byte swizzle).  Launched like prep_tiles_kernel.
__global__ void __launch_bounds__(256) prefill_x16_kernel(const float *x, int M, int K, int BT, int ntt, long chunks,
                                                          uint4 *img) {
    griddep_launch_dependents();
    griddep_wait();
    for (long c = (long)blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += (long)gridDim.x * blockDim.x) {
        const long tile = c / (BT * 8);
        const int within = (int)(c - tile * (BT * 8));
        const int r = within >> 3, pos = within & 7;
        const int kt = (int)(tile / ntt), tt = (int)(tile - (long)kt * ntt);
        const int m = tt * BT + r, k0 = kt * 64 + 8 * (pos ^ (r & 7));
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (m < M && k0 + i < K) ? x[(long)m * K + k0 + i] : 0.0f;
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 p = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            h[i] = *reinterpret_cast<const uint32_t *>(&p);
        }
        img[c] = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// Test hook of the failure detector: one thread waits, through the kernels' bounded wait
// routine, for the first phase of an mbarrier that nothing ever arrives at; after limit_ns
// the wait gives up, sets DEVERR_TIMEOUT in the error word and the kernel returns.
__global__ void wait_expiry_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_wait_limit(b, 0, limit_ns);
}

// The small kernels ask for the same L1 / shared-memory split as the engine (all shared),
// so that an SM does not have to change its configuration between them and the engine and
// they can run beside an engine CTA.  Set once per kernel and device.
static bool prefer_shared(const void *kern) {
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kern, dev})) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return false;
    done.insert({kern, dev});
    return true;
}

int launch_quant_act(const float *x, int M, int K, long ldx, int8_t *xq, float *xd, int32_t *xs, cudaStream_t s) {
    const long blocks = (long)M * (K / 32);
    const int grid = (int)std::min<long>((blocks + 7) / 8, 4096);
    if (!prefer_shared((const void *)quant_act_kernel)) return QG_ECUDA;
    quant_act_kernel<<<grid, 256, 0, s>>>(x, M, K, ldx, xq, xd, xs);
    return cudaGetLastError() == cudaSuccess ? 0 : QG_ECUDA;
}

static int launch_quant_act_s16(const float *x, int M, int K, int16_t *xq, float *xd, int32_t *xs, cudaStream_t s) {
    const long blocks = (long)M * (K / 32);
    const int grid = (int)std::min<long>((blocks + 7) / 8, 4096);
    if (!prefer_shared((const void *)quant_act_s16_kernel)) return QG_ECUDA;
    quant_act_s16_kernel<<<grid, 256, 0, s>>>(x, M, K, xq, xd, xs);
    return cudaGetLastError() == cudaSuccess ? 0 : QG_ECUDA;
}

int launch_splitk_reduce(const float *part, int KS, long MN, float *y, cudaStream_t s) {
    const int grid = (int)std::min<long>((MN + 255) / 256, 1024);
    if (!prefer_shared((const void *)splitk_reduce_kernel)) return QG_ECUDA;
    splitk_reduce_kernel<<<grid, 256, 0, s>>>(part, KS, MN, y);
    return cudaGetLastError() == cudaSuccess ? 0 : QG_ECUDA;
}

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel in the stream is still running (it must griddep_wait() before touching its data).
template <class... KArgs, class... Args>
static int launch_pdl(void (*kern)(KArgs...), int grid, int block, cudaStream_t s, Args... args) {
    if (!prefer_shared((const void *)kern)) return QG_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) != cudaSuccess) return QG_ECUDA;
    return cudaGetLastError() == cudaSuccess ? 0 : QG_ECUDA;
}

int launch_prep_tiles(const float *x, const float *u, float *h_out, const int8_t *xq, const float *xd,
                      const int32_t *xs, int rows, int K, int xgt_log2, uint8_t *img, int8_t *mq, float *md,
                      int32_t *ms, cudaStream_t s) {
    const long blocks = (long)rows * (K / 32);
    const int grid = (int)std::min<long>((blocks + 7) / 8, 2048);
    return launch_pdl(prep_tiles_kernel, grid, 256, s, x, u, h_out, xq, xd, xs, rows, K, xgt_log2, img, mq, md, ms);
}

int launch_prefill_x16(const float *x, int M, int K, int BT, int ntt, int nkt, uint8_t *img, cudaStream_t s) {
    const long chunks = (long)ntt * nkt * BT * 8;
    const int grid = (int)std::min<long>((chunks + 255) / 256, 4096);
    return launch_pdl(prefill_x16_kernel, grid, 256, s, x, M, K, BT, ntt, chunks, reinterpret_cast<uint4 *>(img));
}

int launch_router_prep(const float *x, int M, int H, const float *Wr, int E, float *logits, int xgt_log2,
                       uint8_t *img, bool s16, cudaStream_t s) {
    const long blocks = (long)M * (H / 32);
    const int nprep = (int)std::min<long>((blocks + 7) / 8, 512);
    const int epb = 8 / ROUTER_SPLIT;
    return launch_pdl(router_prep_kernel, (E + epb - 1) / epb + nprep, 256, s, x, M, H, Wr, E, logits, xgt_log2, img,
                      s16);
}

// ----------------------------------------------------------------------------- host helpers
namespace {

struct DevCache {
    std::mutex mu;
    int sms[64] = {};
    int ok[64] = {};  // 0 unknown, 1 supported, -1 not an sm_103 device
};
DevCache g_dev;

// SM count of the current device, or a negative status.
int current_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QG_ECUDA;
    if (dev < 0 || dev >= 64) return QG_EDEVICE;
    std::lock_guard<std::mutex> lock(g_dev.mu);
    if (g_dev.ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QG_ECUDA;
        g_dev.ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        g_dev.sms[dev] = sms;
    }
    return g_dev.ok[dev] == 1 ? g_dev.sms[dev] : QG_EDEVICE;
}

// SM count for planning when no device is usable (workspace queries on any host).
int planning_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
        return sms;
    cudaGetLastError();
    return G_PLAN;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Whether p points into device memory (activations in page-locked host memory are read by
// one preparation kernel, not once per CTA).  The answer is cached per 2 MiB region of the
// address: under unified addressing device and host ranges never share such a region, and
// the answer only chooses between two paths that give the same results, so a stale entry
// (a region freed and reused) costs time at worst.  The query itself takes microseconds.
bool device_memory(const void *p) {
    constexpr int SLOTS = 64;
    static std::mutex mu;
    static uintptr_t key[SLOTS];  // region + 1 (0: empty)
    static bool val[SLOTS];
    const uintptr_t k = ((uintptr_t)p >> 21) + 1;
    const int i = (int)(k % SLOTS);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (key[i] == k) return val[i];
    }
    cudaPointerAttributes a{};
    bool dev = false;
    if (cudaPointerGetAttributes(&a, p) == cudaSuccess)
        dev = a.type == cudaMemoryTypeDevice;
    else
        cudaGetLastError();
    std::lock_guard<std::mutex> lock(mu);
    key[i] = k;
    val[i] = dev;
    return dev;
}

template <class Fn>
int by_format(int fmt, Fn &&fn) {
    switch (fmt) {
    case QG_Q4_0: return fn(std::integral_constant<int, QG_Q4_0>{});
    case QG_Q4_1: return fn(std::integral_constant<int, QG_Q4_1>{});
    case QG_Q5_0: return fn(std::integral_constant<int, QG_Q5_0>{});
    case QG_Q5_1: return fn(std::integral_constant<int, QG_Q5_1>{});
    case QG_IQ4_NL: return fn(std::integral_constant<int, QG_IQ4_NL>{});
    case QG_Q8_0: return fn(std::integral_constant<int, QG_Q8_0>{});
    case QG_Q2_K: return fn(std::integral_constant<int, QG_Q2_K>{});
    case QG_Q3_K: return fn(std::integral_constant<int, QG_Q3_K>{});
    case QG_Q4_K: return fn(std::integral_constant<int, QG_Q4_K>{});
    case QG_Q5_K: return fn(std::integral_constant<int, QG_Q5_K>{});
    case QG_Q6_K: return fn(std::integral_constant<int, QG_Q6_K>{});
    case QG_IQ4_XS: return fn(std::integral_constant<int, QG_IQ4_XS>{});
    default: return QG_EINVAL;
    }
}

bool shape_ok(int fmt, int K) {
    FmtInfo f;
    return fmt_info(fmt, f) && K >= f.qk && K % f.qk == 0;
}

// Fixed scratch of qg_gemv_static_ws: one array per device, shared by every call.
static __device__ __align__(256) uint8_t g_qg_static_ws[QG_STATIC_WS_BYTES];

// The array's address belongs to the context that loaded the module: after a device reset
// (or a host framework that releases and re-creates the primary context) the old address
// is dangling.  The cache is therefore keyed on the current context's unique id, read
// through the driver entry points cuCtxGetCurrent / cuCtxGetId (the runtime API has no
// context id).
typedef CUresult (*PFN_ctx_get_current)(CUcontext *);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long *);

struct StaticWsCache {
    std::mutex mu;
    bool fns_tried = false;
    PFN_ctx_get_current get_current = nullptr;
    PFN_ctx_get_id get_id = nullptr;
    void *addr[64] = {};
    unsigned long long ctx_id[64] = {};
};
StaticWsCache g_static_ws;

// Unique id of the current context, or false if it cannot be read.
bool current_ctx_id(unsigned long long &id) {
    if (!g_static_ws.fns_tried) {
        g_static_ws.fns_tried = true;
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
                cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
            g_static_ws.get_current = reinterpret_cast<PFN_ctx_get_current>(f1);
            g_static_ws.get_id = reinterpret_cast<PFN_ctx_get_id>(f2);
        }
        cudaGetLastError();
    }
    if (!g_static_ws.get_current || !g_static_ws.get_id) return false;
    CUcontext ctx = nullptr;
    if (g_static_ws.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_static_ws.get_id(ctx, &id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context: looked up (cudaGetSymbolAddress)
// on the first call in each context of each device, and again whenever the current context
// of that device has changed since.  Where the context id cannot be read, the address is
// looked up on every call.
void *static_ws_addr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_ws.mu);
    unsigned long long id = 0;
    // before the runtime's first use of the device no context is current yet: the lookup
    // below binds the device's primary context, and its id is read after it
    const bool known = current_ctx_id(id);
    if (known && g_static_ws.addr[dev] && g_static_ws.ctx_id[dev] == id) return g_static_ws.addr[dev];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qg_static_ws) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (current_ctx_id(id)) {
        g_static_ws.addr[dev] = p;
        g_static_ws.ctx_id[dev] = id;
    } else {
        g_static_ws.addr[dev] = nullptr;
    }
    return p;
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" {

int qg_version(void) { return 100; }

const char *qg_strerror(int status) {
    switch (status) {
    case QG_OK: return "ok";
    case QG_EINVAL: return "invalid argument (format, shape, token count, pointer or top-k)";
    case QG_EWORKSPACE: return "workspace missing or smaller than qg_workspace_size()";
    case QG_EALIGN: return "pointer alignment (W and ws: 16 bytes; activations and outputs: 4 bytes)";
    case QG_ECUDA: return "CUDA runtime error or kernel launch failure";
    case QG_EDEVICE: return "current device is not an sm_103 (GB300-class) GPU";
    default: return "unknown status";
    }
}

int qg_quantize_act(const float *x, int M, int K, int8_t *xq, float *xd, int32_t *xs, void *stream) {
    if (!x || !xq || !xd || !xs || M < 1 || K < 32 || K % 32) return QG_EINVAL;
    if (!aligned(x, 4) || !aligned(xd, 4) || !aligned(xs, 4)) return QG_EALIGN;
    const int sms = current_sms();
    if (sms < 0) return sms;
    return launch_quant_act(x, M, K, K, xq, xd, xs, (cudaStream_t)stream);
}

int qg_quantize_act_s16(const float *x, int M, int K, int16_t *xq, float *xd, int32_t *xs, void *stream) {
    if (!x || !xq || !xd || !xs || M < 1 || K < 32 || K % 32) return QG_EINVAL;
    if (!aligned(x, 4) || !aligned(xq, 2) || !aligned(xd, 4) || !aligned(xs, 4)) return QG_EALIGN;
    const int sms = current_sms();
    if (sms < 0) return sms;
    return launch_quant_act_s16(x, M, K, xq, xd, xs, (cudaStream_t)stream);
}

size_t qg_workspace_size(int op, int fmt, int M, int N, int K, int E, int topk, int I) {
    const size_t bad = (size_t)-1;
    switch (op) {
    case QG_OP_GEMV:
    case QG_OP_GEMV_Q: {
        const GemvPlan p = plan_gemv(fmt, N, K, M, planning_sms());
        return p.ok ? p.ws_total : bad;
    }
    case QG_OP_MOE_FFN:
    case QG_OP_MOE_FFN_S16: {
        const MoePlan p = plan_moe(fmt, M, K, E, topk, I, planning_sms(), op == QG_OP_MOE_FFN_S16);
        return p.ok ? p.ws_total : bad;
    }
    case QG_OP_FFN_SUBLAYER: {
        const FfnPlan p = plan_ffn(fmt, M, K, I, planning_sms());
        return p.ok ? p.ws_total : bad;
    }
    case QG_OP_PREFILL: {
        const PrefillPlan p = plan_prefill(fmt, N, K, M, planning_sms());
        return p.ok ? p.ws_total : bad;
    }
    default: return bad;
    }
}

static int gemv_common(int fmt, const void *W, const float *x, const int8_t *xq, const float *xd,
                       const int32_t *xs, float *y, int N, int K, int M, void *ws, size_t ws_bytes, void *stream) {
    if (!W || !y || N < 1 || M < 1 || M > M_MAX || !shape_ok(fmt, K)) return QG_EINVAL;
    if (!x && (!xq || !xd || !xs)) return QG_EINVAL;
    if (!aligned(W, 16) || !aligned(y, 4) || (ws && !aligned(ws, 16))) return QG_EALIGN;
    if (x && !aligned(x, 4)) return QG_EALIGN;
    if (!x && (!aligned(xd, 4) || !aligned(xs, 4))) return QG_EALIGN;
    if (!ws) return QG_EWORKSPACE;
    const int sms = current_sms();
    if (sms < 0) return sms;
    GemvCall c{};
    c.W = static_cast<const uint8_t *>(W);
    c.N = N;
    c.K = K;
    c.M = M;
    c.x = x;
    c.x_device = x && device_memory(x);
    c.xq = x ? nullptr : xq;
    c.xd = x ? nullptr : xd;
    c.xs = x ? nullptr : xs;
    c.y = y;
    c.ws = static_cast<uint8_t *>(ws);
    c.ws_bytes = ws ? ws_bytes : 0;
    c.stream = (cudaStream_t)stream;
    return by_format(fmt, [&](auto F) { return gemv_run<decltype(F)::value>(c, sms); });
}

int qg_gemv(int fmt, const void *W_blocks, const float *x, float *y, int N, int K, int M, void *ws, size_t ws_bytes,
            void *stream) {
    if (!x) return QG_EINVAL;
    return gemv_common(fmt, W_blocks, x, nullptr, nullptr, nullptr, y, N, K, M, ws, ws_bytes, stream);
}

int qg_gemv_static_ws(int fmt, const void *W_blocks, const float *x, float *y, int N, int K, int M, void *stream) {
    if (!x || !W_blocks || !y || N < 1 || M < 1 || M > M_MAX || !shape_ok(fmt, K)) return QG_EINVAL;
    const int sms = current_sms();
    if (sms < 0) return sms;
    const GemvPlan p = plan_gemv(fmt, N, K, M, sms);
    if (!p.ok) return QG_EINVAL;
    if (p.ws_total > (size_t)QG_STATIC_WS_BYTES) return QG_EWORKSPACE;
    void *ws = static_ws_addr();
    if (!ws) return QG_ECUDA;
    return gemv_common(fmt, W_blocks, x, nullptr, nullptr, nullptr, y, N, K, M, ws, QG_STATIC_WS_BYTES, stream);
}

int qg_gemv_q(int fmt, const void *W_blocks, const int8_t *xq, const float *xd, const int32_t *xs, float *y, int N,
              int K, int M, void *ws, size_t ws_bytes, void *stream) {
    if (!xq || !xd || !xs) return QG_EINVAL;
    return gemv_common(fmt, W_blocks, nullptr, xq, xd, xs, y, N, K, M, ws, ws_bytes, stream);
}

int qg_ffn_sublayer(int fmt, const void *Wg, const void *Wu, const void *Wd, const float *x, float *y, int M, int H,
                    int I, void *ws, size_t ws_bytes, void *stream) {
    if (!Wg || !Wu || !Wd || !x || !y || M < 1 || M > M_MAX || !shape_ok(fmt, H) || !shape_ok(fmt, I))
        return QG_EINVAL;
    if (!ws) return QG_EWORKSPACE;
    if (!aligned(Wg, 16) || !aligned(Wu, 16) || !aligned(Wd, 16) || !aligned(ws, 16) || !aligned(x, 4) ||
        !aligned(y, 4))
        return QG_EALIGN;
    const int sms = current_sms();
    if (sms < 0) return sms;
    FfnCall c{};
    c.Wg = static_cast<const uint8_t *>(Wg);
    c.Wu = static_cast<const uint8_t *>(Wu);
    c.Wd = static_cast<const uint8_t *>(Wd);
    c.x = x;
    c.x_device = device_memory(x);
    c.y = y;
    c.M = M;
    c.H = H;
    c.I = I;
    c.ws = static_cast<uint8_t *>(ws);
    c.ws_bytes = ws_bytes;
    c.stream = (cudaStream_t)stream;
    return by_format(fmt, [&](auto F) { return ffn_run<decltype(F)::value>(c, sms); });
}

static int moe_common(bool s16, int fmt, const float *x, int M, int H, const float *Wr, int E, int topk,
                      const void *Wg_exps, const void *Wu_exps, const void *Wd_exps, const void *Wg_sh,
                      const void *Wu_sh, const void *Wd_sh, int I, float *y, int32_t *topk_ids, float *topk_w,
                      void *ws, size_t ws_bytes, void *stream) {
    if (!x || !Wr || !Wg_exps || !Wu_exps || !Wd_exps || !Wg_sh || !Wu_sh || !Wd_sh || !y) return QG_EINVAL;
    if (M < 1 || M > M_MAX || E < 1 || E > E_MAX || topk < 1 || topk > TOPK_MAX || topk > E) return QG_EINVAL;
    if (!shape_ok(fmt, H) || !shape_ok(fmt, I)) return QG_EINVAL;
    if (!ws) return QG_EWORKSPACE;
    const void *w16[] = {Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, ws};
    for (const void *p : w16)
        if (!aligned(p, 16)) return QG_EALIGN;
    if (!aligned(x, 4) || !aligned(Wr, 4) || !aligned(y, 4) || (topk_ids && !aligned(topk_ids, 4)) ||
        (topk_w && !aligned(topk_w, 4)))
        return QG_EALIGN;
    const int sms = current_sms();
    if (sms < 0) return sms;
    MoeCall c{};
    c.x = x;
    c.M = M;
    c.H = H;
    c.Wr = Wr;
    c.E = E;
    c.topk = topk;
    c.Wg_exps = static_cast<const uint8_t *>(Wg_exps);
    c.Wu_exps = static_cast<const uint8_t *>(Wu_exps);
    c.Wd_exps = static_cast<const uint8_t *>(Wd_exps);
    c.Wg_sh = static_cast<const uint8_t *>(Wg_sh);
    c.Wu_sh = static_cast<const uint8_t *>(Wu_sh);
    c.Wd_sh = static_cast<const uint8_t *>(Wd_sh);
    c.I = I;
    c.y = y;
    c.ids_out = topk_ids;
    c.w_out = topk_w;
    c.s16 = s16;
    c.ws = static_cast<uint8_t *>(ws);
    c.ws_bytes = ws_bytes;
    c.stream = (cudaStream_t)stream;
    return by_format(fmt, [&](auto F) { return moe_run<decltype(F)::value>(c, sms); });
}

int qg_moe_ffn(int fmt, const float *x, int M, int H, const float *Wr, int E, int topk, const void *Wg_exps,
               const void *Wu_exps, const void *Wd_exps, const void *Wg_sh, const void *Wu_sh, const void *Wd_sh,
               int I, float *y, int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream) {
    return moe_common(false, fmt, x, M, H, Wr, E, topk, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I, y,
                      topk_ids, topk_w, ws, ws_bytes, stream);
}

int qg_moe_ffn_s16(int fmt, const float *x, int M, int H, const float *Wr, int E, int topk, const void *Wg_exps,
                   const void *Wu_exps, const void *Wd_exps, const void *Wg_sh, const void *Wu_sh, const void *Wd_sh,
                   int I, float *y, int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream) {
    return moe_common(true, fmt, x, M, H, Wr, E, topk, Wg_exps, Wu_exps, Wd_exps, Wg_sh, Wu_sh, Wd_sh, I, y,
                      topk_ids, topk_w, ws, ws_bytes, stream);
}

static int moe_layout(bool s16, int M, int H, int E, int topk, int I, size_t off[7]) {
    if (!off) return QG_EINVAL;
    // the layout does not depend on the block format or the SM count
    const MoePlan p = plan_moe(QG_Q8_0, M, H, E, topk, I, G_PLAN, s16);
    if (!p.ok) return QG_EINVAL;
    off[0] = p.ws_g;
    off[1] = p.ws_u;
    off[2] = p.ws_h;
    off[3] = p.ws_hq;
    off[4] = p.ws_hd;
    off[5] = p.ws_hs;
    off[6] = p.ws_logits;
    return QG_OK;
}

int qg_moe_ws_layout(int M, int H, int E, int topk, int I, size_t off[7]) {
    return moe_layout(false, M, H, E, topk, I, off);
}

int qg_moe_s16_ws_layout(int M, int H, int E, int topk, int I, size_t off[7]) {
    return moe_layout(true, M, H, E, topk, I, off);
}

int qg_ffn_ws_layout(int fmt, int M, int H, int I, size_t off[3]) {
    if (!off) return QG_EINVAL;
    const FfnPlan p = plan_ffn(fmt, M, H, I, G_PLAN);
    if (!p.ok) return QG_EINVAL;
    off[0] = p.ws_g;
    off[1] = p.ws_u;
    off[2] = p.ws_h;
    return QG_OK;
}

int qg_block_dots(int fmt, const void *W, const int8_t *xq, const int32_t *xs, int N, int K, int M, int32_t *dots,
                  int32_t *aux, void *stream) {
    if (!W || !xq || !xs || !dots || !aux || N < 1 || M < 1 || M > M_MAX || !shape_ok(fmt, K)) return QG_EINVAL;
    if (!aligned(W, 16) || !aligned(xs, 4) || !aligned(dots, 4) || !aligned(aux, 4))
        return QG_EALIGN;
    const int sms = current_sms();
    if (sms < 0) return sms;
    DotsCall c{static_cast<const uint8_t *>(W), xq, xs, N, K, M, dots, aux, (cudaStream_t)stream};
    return by_format(fmt, [&](auto F) { return dots_run<decltype(F)::value>(c); });
}

int qg_prefill_gemm(int fmt, const void *W_blocks, const float *x, float *y, int N, int K, int M, void *ws,
                    size_t ws_bytes, void *stream) {
    if (!W_blocks || !x || !y || N < 1 || M < 1 || M > PF_M_MAX || !shape_ok(fmt, K)) return QG_EINVAL;
    if (!aligned(W_blocks, 16) || !aligned(x, 4) || !aligned(y, 4) || (ws && !aligned(ws, 16))) return QG_EALIGN;
    if (!ws) return QG_EWORKSPACE;
    const int sms = current_sms();
    if (sms < 0) return sms;
    const PrefillPlan p = plan_prefill(fmt, N, K, M, sms);
    if (!p.ok) return QG_EINVAL;
    if (ws_bytes < p.ws_total) return QG_EWORKSPACE;
    PrefillCall c{static_cast<const uint8_t *>(W_blocks), x, y, N, K, M, static_cast<uint8_t *>(ws), ws_bytes,
                  (cudaStream_t)stream};
    return by_format(fmt, [&](auto F) { return prefill_run<decltype(F)::value>(c, sms); });
}

int qg_dequant_f16(int fmt, const void *W_blocks, int N, int K, uint16_t *out, void *stream) {
    if (!W_blocks || !out || N < 1 || !shape_ok(fmt, K)) return QG_EINVAL;
    if (!aligned(W_blocks, 16) || !aligned(out, 4)) return QG_EALIGN;
    const int sms = current_sms();
    if (sms < 0) return sms;
    return by_format(fmt, [&](auto F) {
        return dequant_f16_run<decltype(F)::value>(static_cast<const uint8_t *>(W_blocks), N, K, out,
                                                   (cudaStream_t)stream);
    });
}

int qg_test_wait_expiry(unsigned long long limit_ns, void *stream) {
    if (limit_ns < 1000ull || limit_ns > 1000000000ull) return QG_EINVAL;
    const int sms = current_sms();
    if (sms < 0) return sms;
    wait_expiry_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

int qg_device_error(unsigned int *err) {
    if (!err) return QG_EINVAL;
    unsigned int v = 0, zero = 0, all = 0;
    if (cudaMemcpyFromSymbol(&v, g_qg_dev_err, sizeof(v)) != cudaSuccess) return QG_ECUDA;
    if (cudaMemcpyToSymbol(g_qg_dev_err, &zero, sizeof(zero)) != cudaSuccess) return QG_ECUDA;
    all |= v;
    const int fmts[] = {QG_Q4_0, QG_Q4_1, QG_Q5_0, QG_Q5_1, QG_Q8_0, QG_Q2_K, QG_Q3_K,
                        QG_Q4_K, QG_Q5_K, QG_Q6_K, QG_IQ4_NL, QG_IQ4_XS};
    for (int f : fmts) {
        const int rc = by_format(f, [&](auto F) { return dev_err_take<decltype(F)::value>(&v); });
        if (rc) return rc;
        all |= v;
    }
    *err = all;
    return QG_OK;
}

}  // extern "C"
