// qg_engine.cuh -- the weight-streaming engine behind every GEMV-shaped kernel of libqg.
//
// Decode GEMV is bound by HBM bandwidth: every weight byte is read once and used for
// M <= 16 tokens.  The engine therefore spends its effort on keeping enough bytes in
// flight per SM and on never touching a weight byte twice in HBM:
//
//  * one CTA per SM (persistent), NCW consumer warps + 1 producer warp;
//  * the producer's lane 0 copies contiguous runs of raw GGUF blocks from global memory
//    into a ring of S shared-memory slots with 1-D bulk copies (cp.async.bulk, the TMA
//    engine), completion tracked by one mbarrier per slot ("full"); runs that start or
//    end off a 16-byte boundary are widened to it, and the few bytes past the end of a
//    tensor that a widened copy may not read are fetched with byte loads;
//  * consumers wait on "full", decode 32-element units in registers (qg_formats.cuh),
//    multiply with the int8 activation codes by dp4a, apply the fp32 scales, reduce per
//    row inside the warp, and release the slot through an "empty" mbarrier;
//  * per-row partial sums of the warps go to a double-buffered shared array and are
//    added in warp order by the job's epilogue, so every result is deterministic.
//
// A Job supplies the stage sequence (which rows of which tensor each slot receives), the
// activation source, an optional prologue (e.g. quantizing x into shared memory) and the
// epilogue (plain store, split-K partial, SwiGLU, weighted MoE sum).
#pragma once

#include "qg_formats.cuh"

namespace qg {

struct Stage {
    const uint8_t *src[2];  // first byte of each segment (global)
    const uint8_t *lim[2];  // end of the tensor holding segment k: bytes >= lim are never read
    uint32_t bytes[2];      // bytes of each segment
    int nseg;               // 1 or 2 segments
    int R;                  // rows per segment
    uint32_t rstride;       // bytes between consecutive rows of a segment
    int nblk;               // blocks per row
    int xb0;                // activation block of each row's first unit
    int xm;                 // first activation row (token) used by this stage
    int ntok;               // tokens per row (<= MT)
    int tag0, tag1, tag2;   // job-defined
};

// Shared memory carved by the engine (byte offsets from the dynamic smem base).
struct EngineSmem {
    uint32_t ring;   // S slots of slot_bytes (+ STAGE_SLACK each)
    uint32_t part;   // 2 x PART_SLOTS x NCW floats
    uint32_t job;    // job area
    uint32_t bars;   // 2*S mbarriers, then 2*S u32 slot headers (data offsets of the segments)
};

// Shared-memory bytes the engine needs besides the ring and the job area.
__host__ __device__ constexpr uint32_t engine_fixed_smem(int S) {
    return 2u * PART_SLOTS * NCW * 4u + 16u * (uint32_t)S + 8u * (uint32_t)S + 16u;
}

// Sum (in warp order) and clear the partials of stage row i, token m.
template <int MT>
__device__ __forceinline__ float part_take(float *part, int i, int m) {
    float *p = part + (i * MT + m) * NCW;
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
        s += p[w];
        p[w] = 0.0f;
    }
    return s;
}

template <int FMT, int MT, class Job>
__device__ __forceinline__ void process_unit(const Job &job, const typename Job::XSrc &xs, const Stage &st,
                                             uint32_t rowaddr, int u, float (&acc)[MT]) {
    using F = Fmt<FMT>;
    const int b = u / F::UPB, j = u - b * F::UPB;
    WUnit w;
    F::decode(rowaddr + (uint32_t)(b * F::BS), j, w);
    const int xb = st.xb0 + u;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < st.ntok) {
            XUnit x;
            xs.load(st.xm + m, xb, F::NEED_XS, x);
            acc[m] = F::accum(acc[m], w, F::idot(w, x), x);
        }
    }
}

template <int FMT, int MT, class Job>
__global__ void __launch_bounds__(NTHREADS, 1) engine_kernel(const Job job) {
    using F = Fmt<FMT>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int S = job.nslots;
    const uint32_t slot_stride = job.slot_bytes + STAGE_SLACK;

    EngineSmem L;
    L.ring = smem_addr(smem);
    L.part = L.ring + (uint32_t)S * slot_stride;
    L.job = L.part + 2u * PART_SLOTS * NCW * 4u;
    L.bars = L.job + job.job_smem_bytes;
    float *part_base = reinterpret_cast<float *>(smem + (L.part - L.ring));
    uint8_t *job_smem = smem + (L.job - L.ring);
    auto full_bar = [&](int s) { return L.bars + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return L.bars + 8u * (uint32_t)(S + s); };
    auto slot_hdr = [&](int s) { return L.bars + 16u * (uint32_t)S + 8u * (uint32_t)s; };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), NCW);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------------------------------------------ producer
        job.producer_prologue(job_smem, lane);
        __syncwarp();
        if (lane == 0) {
            typename Job::Cursor c;
            job.first(c);
            for (int t = 0; c.valid; ++t, job.next(c)) {
                Stage st;
                job.stage(c, job_smem, true, st);
                const int slot = t % S;
                mbar_wait(empty_bar(slot), (uint32_t)((t / S) & 1) ^ 1u);
                const uint32_t sbase = L.ring + (uint32_t)slot * slot_stride;
                uint32_t off = 0, tx = 0;
                uint32_t cdst[2], cbytes[2];
                const uint8_t *csrc[2];
                for (int k = 0; k < st.nseg; ++k) {
                    const uintptr_t s0 = (uintptr_t)st.src[k];
                    const uintptr_t a0 = s0 & ~(uintptr_t)15;
                    const uintptr_t e = s0 + st.bytes[k];
                    const uintptr_t a1 = (e + 15) & ~(uintptr_t)15;
                    const uintptr_t lim16 = (uintptr_t)st.lim[k] & ~(uintptr_t)15;
                    uintptr_t a1c = a1 <= lim16 ? a1 : lim16;
                    if (a1c < a0) a1c = a0;
                    cdst[k] = sbase + off;
                    csrc[k] = reinterpret_cast<const uint8_t *>(a0);
                    cbytes[k] = (uint32_t)(a1c - a0);
                    tx += cbytes[k];
                    // bytes the widened copy may not read: plain loads
                    for (uintptr_t p = a1c; p < e; ++p)
                        sts8(sbase + off + (uint32_t)(p - a0), *reinterpret_cast<const uint8_t *>(p));
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(slot_hdr(slot) + 4u * k),
                                 "r"(sbase + off + (uint32_t)(s0 & 15)) : "memory");
                    off += (uint32_t)(a1 - a0);
                }
                mbar_arrive_expect_tx(full_bar(slot), tx);
                for (int k = 0; k < st.nseg; ++k)
                    if (cbytes[k]) bulk_g2s(cdst[k], csrc[k], cbytes[k], full_bar(slot));
            }
        }
        return;
    }

    // ---------------------------------------------------------------------- consumers
    for (int i = tid; i < 2 * PART_SLOTS * NCW; i += NCONS) part_base[i] = 0.0f;
    job.consumer_prologue(job_smem, tid);
    consumer_sync();

    const typename Job::XSrc xsrc = job.xsrc(job_smem, L.job);
    typename Job::Cursor c;
    job.first(c);
    int buf = 0;
    for (int t = 0; c.valid; ++t, job.next(c)) {
        Stage st;
        job.stage(c, job_smem, false, st);
        const int slot = t % S;
        float *part = part_base + buf * PART_SLOTS * NCW;
        const int U = st.nblk * F::UPB;
        const int NR = st.nseg * st.R;

        mbar_wait(full_bar(slot), (uint32_t)((t / S) & 1));
        uint32_t data[2];
        data[0] = lds32(slot_hdr(slot));
        data[1] = lds32(slot_hdr(slot) + 4u);

        if (U > 16) {
            const int SPR = (U + 31) >> 5;
            const int TS = NR * SPR;
            const int s0 = warp * TS / NCW, s1 = (warp + 1) * TS / NCW;
            float acc[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
            int cur = -1;
            for (int s = s0; s < s1; ++s) {
                const int i = s / SPR, k = s - i * SPR;
                if (i != cur) {
                    if (cur >= 0) {
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const float v = warp_sum(acc[m]);
                            if (lane == 0) part[(cur * MT + m) * NCW + warp] = v;
                            acc[m] = 0.0f;
                        }
                    }
                    cur = i;
                }
                const int u = 32 * k + lane;
                if (u < U) {
                    const int sg = i >= st.R;
                    const uint32_t rowaddr = data[sg] + (uint32_t)(i - sg * st.R) * st.rstride;
                    process_unit<FMT, MT>(job, xsrc, st, rowaddr, u, acc);
                }
            }
            if (cur >= 0) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float v = warp_sum(acc[m]);
                    if (lane == 0) part[(cur * MT + m) * NCW + warp] = v;
                }
            }
        } else {
            // short rows: 32/Up rows per warp step, Up = U rounded up to a power of two
            int Up = 1;
            while (Up < U) Up <<= 1;
            const int P = 32 / Up;
            const int TS = (NR + P - 1) / P;
            const int s0 = warp * TS / NCW, s1 = (warp + 1) * TS / NCW;
            for (int s = s0; s < s1; ++s) {
                const int i = s * P + lane / Up, u = lane & (Up - 1);
                float acc[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
                if (u < U && i < NR) {
                    const int sg = i >= st.R;
                    const uint32_t rowaddr = data[sg] + (uint32_t)(i - sg * st.R) * st.rstride;
                    process_unit<FMT, MT>(job, xsrc, st, rowaddr, u, acc);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v = acc[m];
                    for (int o = Up >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (u == 0 && i < NR) part[(i * MT + m) * NCW + warp] = v;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(slot));
        consumer_sync();
        job.template epilogue<MT>(st, part, job_smem, tid);
        buf ^= 1;
    }
}

}  // namespace qg
