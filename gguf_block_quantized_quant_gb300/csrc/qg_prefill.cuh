// qg_prefill.cuh -- prefill GEMM over raw GGUF blocks on the 5th-generation tensor cores.
//
// "01 · 阶段总览：从 2B 到 8B 再到 MoE", section 九: once decode is bound by memory, prefill (M
// tokens at once, M >> 16) is a dense contraction, and the page moved it to the tensor cores
// with the weights dequantized to fp16 inside the kernel (prefill of 512 tokens 372 -> 902
// tokens/s); section 四, issue ⑮: prefill takes float activations, not int8 ones.  So
//     y[m][n] = sum_k fp16(w[n][k]) * fp16(x[m][k]),   accumulated in fp32,
// with w formed per 32-element unit as in qg_dequant.cuh and x rounded to fp16 by a small
// preparation kernel that writes the activation tiles in the tensor cores' operand layout.
//
// One CTA computes a tile of 128 weight rows x NT token tiles of BT tokens (BT <= 256, NT 1
// or 2: each dequantized weight tile then serves up to 512 tokens) over a range of K:
//   * warps 0-7 (dequant): thread t owns row t % 128 and, per K step of 64, the unit t / 128
//     (32 elements); it fetches the raw words of the unit two steps ahead, converts them to
//     fp16 and stores them as four 16-byte chunks of the swizzled weight tile of the stage;
//   * warp 8 lane 0 (producer): one 1-D bulk copy per stage of the activation tile
//     (NT tiles of BT rows x 128 bytes, adjacent in the image and laid out by the preparation
//     kernel exactly as they must sit in shared memory); warp 8 also allocates and frees the
//     tensor memory;
//   * warp 9 lane 0 (MMA): per stage and token tile, four tcgen05.mma of M = 128, N = BT,
//     K = 16 into that tile's fp32 accumulator in tensor memory (128 lanes x BT columns each),
//     then tcgen05.commit to the stage's "empty" barrier, which frees the stage for both
//     producers;
//   * after the last stage the MMA thread commits to "done"; warps 0-7 read the accumulator
//     with tcgen05.ld (warp w: lanes 32 (w % 4) .., half of the columns) and write y (or a
//     K-slice's partial sums, added by the split-K reduction).
// Every wait is bounded; after one gives up the kernel still runs to its end, waits (again
// bounded) for its own bulk copies and MMAs, and frees its tensor memory.
#pragma once

#include "qg_dequant.cuh"
#include "qg_umma.h"

namespace qg {

constexpr int PF_DEQ_WARPS = 8;
constexpr int PF_THREADS = (PF_DEQ_WARPS + 2) * 32;
constexpr int PF_LOOKAHEAD = 2;           // K steps whose raw words a dequant thread holds ahead

struct PrefillArgs {
    const uint8_t *W;
    uint32_t rb;          // bytes per weight row
    int N, K, M;
    int BT;               // tokens per token tile (MMA N): a multiple of 16, at most 256
    int NT;               // token tiles per CTA (1 or 2)
    int ntt;              // token tiles of the whole batch
    int nkt;              // K tiles of 64 (the last one zero-padded when K % 64 == 32)
    int ktps;             // K tiles per K-slice (blockIdx.z)
    int stages;
    int tmem_cols;
    uint32_t idesc;
    const uint8_t *ximg;  // [K tile][token tile][BT x 128 bytes]
    float *out;           // y, or partials [KS][M][N]
};

__host__ __device__ constexpr uint32_t prefill_stage_bytes(int BT, int NT) {
    return (uint32_t)(PF_BM * 128 + NT * BT * 128);
}
__host__ __device__ constexpr uint32_t prefill_smem_bytes(int BT, int NT, int stages) {
    return (uint32_t)stages * prefill_stage_bytes(BT, NT) + UMMA_ATOM_BYTES /* alignment slack */ +
           8u * (uint32_t)(3 * stages + 1) + 16u;
}

// ------------------------------------------------------------------ tcgen05 wrappers
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (tensor memory) = A * B^T (+ D when accumulate), A and B K-major in shared memory.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}
// The barrier's phase completes (one arrival) when every tcgen05.mma issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 16 consecutive fp32 columns of the warp's 32 lanes: v[i] = column col + i of lane (lane
// quarter of the address) + laneid.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

template <int FMT>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_kernel(const PrefillArgs a) {
    using D = Deq<FMT>;
    extern __shared__ __align__(16) uint8_t pf_smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.stages;
    const uint32_t wtile = PF_BM * 128, ttile = (uint32_t)a.BT * 128, xtile = (uint32_t)a.NT * ttile;
    const uint32_t base = (smem_addr(pf_smem) + (UMMA_ATOM_BYTES - 1)) & ~(UMMA_ATOM_BYTES - 1);
    const uint32_t wt0 = base, xt0 = base + (uint32_t)S * wtile;
    const uint32_t bars = xt0 + (uint32_t)S * xtile;
    auto xfull = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto wfull = [&](int s) { return bars + 8u * (uint32_t)(S + s); };
    auto empty = [&](int s) { return bars + 8u * (uint32_t)(2 * S + s); };
    const uint32_t done = bars + 8u * (uint32_t)(3 * S);
    const uint32_t taddr_slot = done + 8u;

    const int n0 = (int)blockIdx.x * PF_BM, tt0 = (int)blockIdx.y * a.NT, ks = (int)blockIdx.z;
    const int ntc = min(a.NT, a.ntt - tt0);  // token tiles of this CTA
    const int kt0 = ks * a.ktps;
    const int nk = min(a.nkt, kt0 + a.ktps) - kt0;  // >= 1 by the plan

    griddep_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(xfull(s), 1);
            mbar_init(wfull(s), PF_DEQ_WARPS * 32);
            mbar_init(empty(s), 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == PF_DEQ_WARPS) tmem_alloc(taddr_slot, (uint32_t)a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = lds32(taddr_slot);
    // the activation image comes from the preceding kernel (and, through its own wait,
    // everything before it is complete too)
    griddep_wait();

    if (warp < PF_DEQ_WARPS) {
        // ------------------------------------------------------------ dequant warps
        const int r = tid & (PF_BM - 1), hsel = tid >> 7;
        const int n = n0 + r;
        const bool row_ok = n < a.N;
        const uint8_t *row = a.W + (size_t)(row_ok ? n : 0) * a.rb;
        const uint8_t *lim = a.W + (size_t)a.N * a.rb;  // end of the tensor
        const int nunits = a.K / 32;
        typename D::Raw raw[PF_LOOKAHEAD + 1];
        auto fetch = [&](int i, typename D::Raw &rw) {
            const int u = 2 * (kt0 + i) + hsel;
            if (row_ok && i < nk && u < nunits) D::fetch(row, u, lim, rw);
        };
#pragma unroll
        for (int p = 0; p < PF_LOOKAHEAD; ++p) fetch(p, raw[p]);
        for (int i = 0; i < nk; ++i) {
            fetch(i + PF_LOOKAHEAD, raw[PF_LOOKAHEAD]);
            const int s = i % S;
            if (i >= S) mbar_wait(empty(s), (uint32_t)((i / S - 1) & 1));
            const int u = 2 * (kt0 + i) + hsel;
            uint32_t h[16];
            if (row_ok && u < nunits) {
                deq_convert<FMT>(raw[0], u, h);
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) h[q] = 0u;  // rows past N, K past its end
            }
            const uint32_t rbase = wt0 + (uint32_t)s * wtile + (uint32_t)r * 128u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t cc = (uint32_t)(4 * hsel + c);
                sts128(rbase + ((cc ^ ((uint32_t)r & 7u)) << 4), h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
            }
            fence_proxy_async_smem();  // the tensor cores read the tile through the async proxy
            mbar_arrive(wfull(s));
#pragma unroll
            for (int p = 0; p < PF_LOOKAHEAD; ++p)
#pragma unroll
                for (int q = 0; q < D::RW; ++q) raw[p][q] = raw[p + 1][q];
        }
    } else if (warp == PF_DEQ_WARPS) {
        // ------------------------------------------------------------ activation producer
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)ntc * ttile;
            for (int i = 0; i < nk; ++i) {
                const int s = i % S;
                if (i >= S) mbar_wait(empty(s), (uint32_t)((i / S - 1) & 1));
                mbar_arrive_expect_tx(xfull(s), bytes);
                bulk_g2s(xt0 + (uint32_t)s * xtile, a.ximg + ((size_t)(kt0 + i) * a.ntt + tt0) * ttile, bytes,
                         xfull(s));
            }
        }
    } else {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int i = 0; i < nk; ++i) {
                const int s = i % S;
                const uint32_t ph = (uint32_t)((i / S) & 1);
                mbar_wait(wfull(s), ph);
                mbar_wait(xfull(s), ph);
                tc_fence_after();
                const uint64_t ad = umma_desc_kmajor_sw128(wt0 + (uint32_t)s * wtile);
                for (int t = 0; t < ntc; ++t) {
                    const uint64_t bd = umma_desc_kmajor_sw128(xt0 + (uint32_t)s * xtile + (uint32_t)t * ttile);
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the row
                        umma_f16(tmem + (uint32_t)(t * a.BT), ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk),
                                 a.idesc, (i | kk) != 0);
                }
                umma_commit(empty(s));
            }
            umma_commit(done);
        }
    }

    if (warp < PF_DEQ_WARPS) {
        // ------------------------------------------------------------ epilogue
        mbar_wait(done, 0);
        tc_fence_after();
        const int q = warp & 3, hf = warp >> 2;
        const int cols = ntc * a.BT;  // token columns of the CTA's accumulators
        const int split = ((cols / 2 + 15) / 16) * 16;
        const int c0 = hf ? split : 0, c1 = hf ? cols : split;
        const int n = n0 + 32 * q + lane;
        float *out = a.out + (size_t)ks * a.M * a.N;
        for (int c = c0; c < c1; c += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c, v);
            if (n < a.N) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = tt0 * a.BT + c + j;
                    if (m < a.M) out[(size_t)m * a.N + n] = __uint_as_float(v[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == PF_DEQ_WARPS) {
        tc_fence_after();
        if (lane == 0) {
            // normally complete already; after a timeout, let in-flight copies and MMAs end
            // before the shared and tensor memory they target are released
            for (int s = 0; s < S && s < nk; ++s) {
                const int ilast = s + S * ((nk - 1 - s) / S);
                mbar_drain(xfull(s), (uint32_t)((ilast / S) & 1), DRAIN_NS);
            }
            mbar_drain(done, 0, DRAIN_NS);
        }
        __syncwarp();
        tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
    }
}

// fp16 weights of whole rows, through the same unit decoders (test hook): thread per
// (row, unit), 32 values written as 64 bytes.
template <int FMT>
__global__ void __launch_bounds__(256) dequant_f16_kernel(const uint8_t *W, uint32_t rb, int N, int K, uint16_t *out) {
    using D = Deq<FMT>;
    const int nu = K / 32;
    const long total = (long)N * nu;
    for (long t = (long)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (long)gridDim.x * blockDim.x) {
        const int n = (int)(t / nu), u = (int)(t % nu);
        typename D::Raw raw;
        D::fetch(W + (size_t)n * rb, u, W + (size_t)N * rb, raw);
        uint32_t h[16];
        deq_convert<FMT>(raw, u, h);
        uint32_t *o = reinterpret_cast<uint32_t *>(out + (size_t)n * K + 32 * u);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = h[i];
    }
}

}  // namespace qg
