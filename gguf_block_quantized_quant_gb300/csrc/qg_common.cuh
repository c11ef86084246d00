// qg_common.cuh -- device helpers shared by the libqg kernels: shared-memory loads,
// mbarrier / 1-D bulk-copy (TMA) wrappers with bounded waits, warp reductions and the
// per-32 activation quantizer.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qg {

// ---------------------------------------------------------------------------------
// Launch geometry of the streaming engine: engine_ncw() warps, one CTA per SM.  A lane
// copies its task from the ring into registers before decoding it, so a ring slot is busy
// only until then.  Tasks of at most 160 bytes with up to 4 tokens per lane run 16 warps
// (4 per scheduler, to hide the latency of the decode chains); larger tasks hold up to 72
// words per lane and run 8 warps with the room of two ring slots each, as do 8 or 16
// tokens per lane (more accumulator registers).
__host__ __device__ constexpr int engine_ncw(int task_bytes, int MT) {
    return (MT <= 4 && task_bytes <= 160) ? 16 : 8;
}
// One-token launches with tasks over 160 bytes may run 12 warps (3 per scheduler) with one
// ring slot each when every CTA has enough tasks for two stages per warp.
constexpr int NCW_WIDE = 12;
__host__ __device__ constexpr bool ncw_wide_allowed(int task_bytes, int MT) { return MT == 1 && task_bytes > 160; }

constexpr int SMEM_MAX = 227 * 1024;       // opt-in dynamic shared memory per CTA (sm_100 family)
constexpr int STAGE_SLACK = 64;            // bytes after each ring slot for over-reads

// Device error word: bit 0 = a bounded wait gave up; bit 1 = a stage did not fit the
// engine's piece table (its remaining tasks were skipped).
constexpr unsigned int DEVERR_TIMEOUT = 1u;
constexpr unsigned int DEVERR_PLAN = 2u;
constexpr unsigned long long WAIT_NS = 2000000000ull;   // 2 s
constexpr unsigned long long WAIT_CHECK_NS = 1000000ull; // 1 ms: look for an earlier timeout

// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts8(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ldg128_nc(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// byte select: result byte n = byte ((sel >> 4n) & 7) of the 8-byte value {b:a}.
// The selector's bit 3 of each nibble is always clear at every call site.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h16) {
    return __half2float(__ushort_as_half((unsigned short)(h16 & 0xffffu)));
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a((int)a, (int)b, c);
}

// ---------------------------------------------------------------------------------
// mbarrier + bulk copy (PTX ISA 8.x, sm_90+)
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// The bulk copies of a stage may complete before the issuing lane posts their byte count: the
// transaction count may go negative until then, and the phase cannot complete before the
// issuing lane's arrival.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Potentially blocking test: the thread may be suspended (up to about WAIT_HINT_NS) until
// the phase completes, instead of spinning.
constexpr uint32_t WAIT_HINT_NS = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(WAIT_HINT_NS)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the phase of parity `parity` (for polling several barriers).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One error word per translation unit (no relocatable device code); the host ORs them.
static __device__ unsigned int g_qg_dev_err;

// Waits for the phase of parity `parity` to complete.  Gives up after limit_ns, records
// DEVERR_TIMEOUT in the device error word and returns false; the caller then carries on
// (with invalid data) so that every thread still reaches every barrier and the kernel
// ends.  The host reads the error word through qg_device_error().
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    bool checked = false;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            const unsigned long long dt = globaltimer_ns() - t0;
            // a wait this long is abnormal: if another wait already gave up, the data is
            // invalid anyway, so do not wait again (read once; off the normal path)
            if (!checked && dt > WAIT_CHECK_NS) {
                checked = true;
                if (*reinterpret_cast<volatile unsigned int *>(&g_qg_dev_err) & DEVERR_TIMEOUT) return false;
            }
            if (dt > limit_ns) {
                atomicOr(&g_qg_dev_err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}
// The kernels' wait: limit WAIT_NS.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) { return mbar_wait_limit(bar, parity, WAIT_NS); }

// Waits for the phase of parity `parity` of `bar` for at most limit_ns, without looking at
// the device error word.  For the end of a kernel: after an earlier wait gave up, bulk copies
// (or tensor-core operations) still in flight must land before the shared or tensor memory
// they target is released.  On the normal path the phase is complete and this returns at
// once.  Returns whether the phase completed.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}
constexpr unsigned long long DRAIN_NS = 100000000ull;  // 100 ms

// 1-D bulk copy global -> shared (this CTA), completion counted on `bar` in bytes.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Programmatic dependent launch: a kernel launched with the programmatic-serialization
// attribute may start before the previous kernel in the stream has finished; it must call
// griddep_wait() before reading anything that kernel writes.  The previous kernel calls
// griddep_launch_dependents() to let it start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Barrier among the NCONS threads that reach it (every warp of the engine).
template <int NCONS>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NCONS) : "memory");
}

// ---------------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Activation quantization of one 32-element block by one warp: lane i holds element i.
// d = amax/127 (IEEE fp32 division), q = clamp(roundf(v/d)) (half away from zero).
__device__ __forceinline__ void quant_block_warp(float v, int &q, float &d, int &s) {
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    d = __fdiv_rn(a, 127.0f);
    q = 0;
    if (d != 0.0f) {
        q = (int)roundf(__fdiv_rn(v, d));
        q = q > 127 ? 127 : (q < -127 ? -127 : q);
    }
    s = __reduce_add_sync(0xffffffffu, q);
}

// s16 activation quantization of one 32-element block, one element per lane: the same
// rule with a step 256 times finer, d = amax / 32512 (= (amax / 127) / 256) and codes in
// [-32512, 32512].
constexpr int S16_QMAX = 127 * 256;
__device__ __forceinline__ void quant_block_warp16(float v, int &q, float &d, int &s) {
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    d = __fdiv_rn(a, (float)S16_QMAX);
    q = 0;
    if (d != 0.0f) {
        q = (int)roundf(__fdiv_rn(v, d));
        q = q > S16_QMAX ? S16_QMAX : (q < -S16_QMAX ? -S16_QMAX : q);
    }
    s = __reduce_add_sync(0xffffffffu, q);
}

}  // namespace qg
