// prefill_model.cu -- host checks of the prefill GEMM's launch plans and tensor-core
// descriptors, run on the CPU before any GPU launch (tests/test_prefill_host.py).
//
// 1. Descriptors: the shared-memory and instruction descriptors are decoded field by field
//    with the documented bit positions (written out here again, independently of qg_umma.h)
//    and compared with the intended values.
// 2. The 128-byte swizzle used by the producers: sw128_offset is a bijection of each
//    1024-byte atom and agrees with the chunk-position rule of the activation image kernel
//    (position p of row r holds logical chunk p ^ (r & 7)).
// 3. Plans over a sweep of shapes and every block format: tile shape within the MMA's
//    limits, tensor-memory columns, shared memory, every K-slice non-empty; for every CTA:
//    the activation copies stay inside the workspace image, the outputs inside y or the
//    partial-sum buffer, and every weight fetch of every unit stays inside its row with the
//    alignment of the load that reads it.
// Prints "fails 0" when every check holds.
#include <cstdio>
#include <vector>

#include "qg_plan.h"
using namespace qg;

static int fails = 0;
#define CHECK(c, ...)                                   \
    do {                                                \
        if (!(c)) {                                     \
            ++fails;                                    \
            if (fails < 30) {                           \
                printf("FAIL %d: ", __LINE__);          \
                printf(__VA_ARGS__);                    \
                printf("\n");                           \
            }                                           \
        }                                               \
    } while (0)

static uint64_t bits(uint64_t v, int lo, int hi) { return (v >> lo) & ((1ull << (hi - lo + 1)) - 1); }

static void check_descriptors() {
    for (uint32_t addr = 0; addr < (1u << 18); addr += 1024) {
        const uint64_t d = umma_desc_kmajor_sw128(addr);
        CHECK(bits(d, 0, 13) == (addr >> 4), "start field %u", addr);
        CHECK(bits(d, 14, 15) == 0, "bits 14-15");
        CHECK(bits(d, 16, 29) == 1, "leading byte offset field (16 bytes)");
        CHECK(bits(d, 30, 31) == 0, "bits 30-31");
        CHECK(bits(d, 32, 45) == 1024 / 16, "stride byte offset field (1024 bytes)");
        CHECK(bits(d, 46, 48) == 1, "fixed 0b001 at bits 46-48");
        CHECK(bits(d, 49, 51) == 0, "base offset");
        CHECK(bits(d, 52, 52) == 0, "leading-dimension mode");
        CHECK(bits(d, 53, 60) == 0, "bits 53-60");
        CHECK(bits(d, 61, 63) == 2, "swizzle mode 128B = 2");
        // advancing K by 16 fp16 (32 bytes) moves only the start field, by 2
        for (int kk = 0; kk < 4; ++kk) CHECK(d + 2 * kk == umma_desc_kmajor_sw128(addr + 32 * kk), "K advance");
    }
    for (int n = 16; n <= 256; n += 16) {
        const uint32_t i = umma_idesc_f16(128, n);
        CHECK(bits(i, 0, 3) == 0, "sparsity/saturate");
        CHECK(bits(i, 4, 5) == 1, "D type fp32");
        CHECK(bits(i, 6, 6) == 0, "bit 6");
        CHECK(bits(i, 7, 9) == 0 && bits(i, 10, 12) == 0, "A, B fp16");
        CHECK(bits(i, 13, 14) == 0, "no negation");
        CHECK(bits(i, 15, 16) == 0, "A, B K-major");
        CHECK(bits(i, 17, 22) == (uint32_t)(n >> 3), "N >> 3 at bits 17-22");
        CHECK(bits(i, 23, 23) == 0, "bit 23");
        CHECK(bits(i, 24, 28) == 128 >> 4, "M >> 4 at bits 24-28");
        CHECK(bits(i, 29, 31) == 0, "bits 29-31");
        CHECK(umma_shape_ok(128, n), "shape %d", n);
        const int cols = tmem_cols_for(n);
        CHECK(cols >= n && cols >= 32 && (cols & (cols - 1)) == 0 && cols <= 512, "tmem cols %d for %d", cols, n);
    }
}

static void check_swizzle() {
    // sw128_offset maps (r, k) of an 8-row atom onto distinct 2-byte slots of 1024 bytes
    std::vector<int> seen(512, 0);
    for (uint32_t r = 0; r < 8; ++r)
        for (uint32_t k = 0; k < 64; ++k) {
            const uint32_t o = sw128_offset(r, k);
            CHECK(o < 1024 && o % 2 == 0, "offset %u", o);
            if (o < 1024) seen[o / 2]++;
            // the image kernel: position p holds logical chunk p ^ (r & 7)
            const uint32_t p = (o % 128) / 16;
            CHECK((p ^ (r & 7)) == k / 8 && o / 128 == r && (o % 16) / 2 == k % 8, "image rule r %u k %u", r, k);
        }
    for (int i = 0; i < 512; ++i) CHECK(seen[i] == 1, "slot %d seen %d", i, seen[i]);
}

// Byte ranges (offset from the row start, size, alignment of the load) that unit u's fetch
// reads, mirroring each format's fetch() in qg_dequant.cuh.
struct Rd {
    long off;
    int size, align;
};
static std::vector<Rd> fetch_reads(int fmt, int u) {
    std::vector<Rd> v;
    FmtInfo f;
    fmt_info(fmt, f);
    auto add = [&](long off, int size, int align) { v.push_back({off, size, align}); };
    if (f.qk == 32) {
        // legacy blocks: read by fetch_words through the aligned 16-byte chunks covering the
        // block (checked separately, check_legacy_windows); the slow path near the tensor's
        // end reads the block's own 16-bit units
        const long b = (long)u * f.bs;
        for (int i = 0; i < f.bs / 2; ++i) add(b + 2 * i, 2, 2);
        return v;
    }
    const long b = (long)(u / 8) * f.bs;
    const int j = u % 8, hh = j / 4;
    switch (fmt) {
    case 10:  // Q2_K
        add(b + 2 * j, 2, 2);
        add(b + 80, 4, 4);
        for (int i = 0; i < 8; ++i) add(b + 16 + 32 * hh + 4 * i, 4, 4);
        break;
    case 11:  // Q3_K
        for (int i = 0; i < 8; ++i) add(b + 4 * i, 4, 2);
        for (int i = 0; i < 8; ++i) add(b + 32 + 32 * hh + 4 * i, 4, 2);
        add(b + 96 + (2 * j) % 8, 2, 2);
        add(b + 104 + (2 * j) % 4, 2, 2);
        add(b + 108, 2, 2);
        break;
    case 12:
    case 13: {  // Q4_K, Q5_K: 16-byte loads
        const bool q5 = fmt == 13;
        add(b, 16, 16);
        add(b + (q5 ? 48 : 16) + 32 * (j / 2), 16, 16);
        add(b + (q5 ? 48 : 16) + 32 * (j / 2) + 16, 16, 16);
        if (q5) {
            add(b + 16, 16, 16);
            add(b + 32, 16, 16);
        }
        break;
    }
    case 14:  // Q6_K
        for (int i = 0; i < 8; ++i) add(b + 64 * hh + 32 * ((j % 4) & 1) + 4 * i, 4, 2);
        for (int i = 0; i < 8; ++i) add(b + 128 + 32 * hh + 4 * i, 4, 2);
        add(b + 192 + 2 * j, 2, 2);
        add(b + 208, 2, 2);
        break;
    case 23:  // IQ4_XS
        add(b, 4, 4);
        add(b + 4, 4, 4);
        for (int i = 0; i < 4; ++i) add(b + 8 + 16 * j + 4 * i, 4, 4);
        break;
    }
    return v;
}

static long gcd_l(long a, long b) { return b ? gcd_l(b, a % b) : a; }

static void check_fetches(int fmt, int K) {
    FmtInfo f;
    fmt_info(fmt, f);
    const long rb = (long)(K / f.qk) * f.bs;
    const long row_align = gcd_l(rb, 16);  // rows start at multiples of rb from a 16-byte-aligned tensor
    for (int u = 0; u < K / 32; ++u)
        for (const Rd &r : fetch_reads(fmt, u)) {
            CHECK(r.off >= 0 && r.off + r.size <= rb, "fmt %d K %d unit %d reads [%ld, %ld) of a %ld-byte row", fmt,
                  K, u, r.off, r.off + r.size, rb);
            CHECK(row_align % r.align == 0 && r.off % r.align == 0, "fmt %d K %d unit %d: load of %d bytes at %ld "
                  "needs %d-byte alignment (rows %ld-aligned)", fmt, K, u, r.size, r.off, r.align, row_align);
            // every unit reads inside its own block
            const long blk = (long)(u / (f.qk / 32)) * f.bs;
            CHECK(r.off >= blk && r.off + r.size <= blk + f.bs, "fmt %d unit %d read outside its block", fmt, u);
        }
}

// fetch_words of the 32-element block formats over a tensor of N rows: the covering window
// of NC chunks (MAXO = the largest offset of a block within its first chunk) holds every byte
// of the block, and is only read when it lies inside the tensor.
static void check_legacy_windows(int fmt, int K, int N) {
    FmtInfo f;
    fmt_info(fmt, f);
    if (f.qk != 32) return;
    const int maxo = fmt == 7 ? 8 : fmt == 3 ? 12 : 14;
    const int nc = (maxo + f.bs + 15) / 16;
    const long rb = (long)(K / 32) * f.bs, end = (long)N * rb;
    for (int n = 0; n < N; ++n)
        for (int u = 0; u < K / 32; ++u) {
            const long p = (long)n * rb + (long)u * f.bs;  // tensor offsets (the tensor is 16-byte aligned)
            const long base = p & ~15L, o = p - base;
            CHECK(p % 2 == 0, "fmt %d block offset %ld odd", fmt, p);
            CHECK(o <= maxo, "fmt %d K %d block offset %ld in its chunk > %d", fmt, K, o, maxo);
            CHECK(o + f.bs <= 16L * nc, "fmt %d window of %d chunks misses block bytes", fmt, nc);
            if (base + 16L * nc <= end) CHECK(base >= 0 && base % 16 == 0, "fmt %d window", fmt);
        }
}

static void check_plan(int fmt, int N, int K, int M, int sms) {
    const PrefillPlan p = plan_prefill(fmt, N, K, M, sms);
    CHECK(p.ok, "plan fmt %d N %d K %d M %d not ok", fmt, N, K, M);
    if (!p.ok) return;
    CHECK(p.BT % 16 == 0 && p.BT >= 16 && p.BT <= 256 && umma_shape_ok(PF_BM, p.BT), "BT %d", p.BT);
    CHECK(p.BT >= 256 || p.BT >= M, "BT %d < M %d", p.BT, M);
    CHECK(p.NT >= 1 && p.NT <= 2 && p.NT <= p.ntt && p.ngrp == (p.ntt + p.NT - 1) / p.NT, "NT %d ngrp %d", p.NT, p.ngrp);
    CHECK(p.tmem_cols >= p.NT * p.BT && p.tmem_cols <= 512 && (p.tmem_cols & (p.tmem_cols - 1)) == 0, "tmem cols %d",
          p.tmem_cols);
    CHECK(p.idesc == umma_idesc_f16(PF_BM, p.BT), "idesc");
    CHECK(p.stages >= 2 && p.smem <= (uint32_t)SMEM_MAX, "stages %d smem %u", p.stages, p.smem);
    // the kernel's layout inside its dynamic shared memory (worst-case alignment slack)
    const uint32_t used = (UMMA_ATOM_BYTES - 16) + (uint32_t)p.stages * prefill_stage_bytes(p.BT, p.NT) +
                          8u * (uint32_t)(3 * p.stages) + 8u + 4u;
    CHECK(used <= p.smem, "smem layout %u > %u", used, p.smem);
    CHECK(prefill_stage_bytes(p.BT, p.NT) % UMMA_ATOM_BYTES == 0 && (p.BT * 128) % UMMA_ATOM_BYTES == 0,
          "tiles keep 1024-byte alignment");
    CHECK(p.nn == (N + 127) / 128 && p.ntt == (M + p.BT - 1) / p.BT && p.nkt == (K + 63) / 64, "grid");
    CHECK(p.ngrp <= 65535 && p.KS <= 65535, "grid y/z");
    CHECK(p.KS >= 1 && p.ktps >= 1 && (long)p.KS * p.ktps >= p.nkt && (long)(p.KS - 1) * p.ktps < p.nkt,
          "slices KS %d ktps %d nkt %d", p.KS, p.ktps, p.nkt);
    const size_t img = (size_t)p.ntt * p.nkt * p.BT * 128;
    CHECK(p.ws_ximg + img <= p.ws_total, "image in workspace");
    if (p.KS > 1) CHECK(p.ws_part >= p.ws_ximg + img && p.ws_part + 4ull * p.KS * M * N <= p.ws_total, "partials");
    CHECK(p.ws_ximg % 256 == 0 && p.ws_part % 16 == 0, "workspace alignment");
    // every CTA: its copies (K tile major image: a stage copies the CTA's ntc adjacent token
    // tiles of one K tile) and its outputs
    for (int ks = 0; ks < p.KS; ++ks) {
        const int kt0 = ks * p.ktps, nk = std::min(p.nkt, kt0 + p.ktps) - kt0;
        CHECK(nk >= 1, "empty slice");
        for (int gy = 0; gy < p.ngrp; ++gy) {
            const int tt0 = gy * p.NT, ntc = std::min(p.NT, p.ntt - tt0);
            CHECK(ntc >= 1, "empty token group");
            for (int i = 0; i < nk; ++i) {
                const size_t off = ((size_t)(kt0 + i) * p.ntt + tt0) * p.BT * 128, bytes = (size_t)ntc * p.BT * 128;
                CHECK(off + bytes <= img && bytes <= (size_t)p.NT * p.BT * 128, "activation copy of CTA (%d, %d) stage %d",
                      gy, ks, i);
            }
            const long m_hi = std::min<long>(M, (long)(tt0 + ntc) * p.BT) - 1;
            const size_t out_hi = (size_t)ks * M * N + (size_t)m_hi * N + (N - 1);
            CHECK(out_hi < (size_t)(p.KS > 1 ? p.KS : 1) * M * N, "output index");
            // accumulator columns: ntc tiles of BT columns inside the allocation
            CHECK(ntc * p.BT <= p.tmem_cols, "accumulator columns");
        }
    }
    // the epilogue's column split: multiples of 16 covering [0, ntc * BT)
    for (int ntc = 1; ntc <= p.NT; ++ntc) {
        const int cols = ntc * p.BT, split = ((cols / 2 + 15) / 16) * 16;
        CHECK(split % 16 == 0 && split <= cols && (cols - split) % 16 == 0, "epilogue split %d of %d", split, cols);
    }
}

int main() {
    check_descriptors();
    check_swizzle();
    const int fmts[] = {2, 3, 6, 7, 8, 10, 11, 12, 13, 14, 20, 23};
    long plans = 0;
    for (int fmt : fmts) {
        FmtInfo f;
        fmt_info(fmt, f);
        for (int K : {f.qk, 2 * f.qk, 3 * f.qk, 1024, 2048, 4096, 5120, 17408, 96 * f.qk}) {
            check_fetches(fmt, K);
            for (int N : {1, 2, 3, 7}) check_legacy_windows(fmt, K, N);
        }
        for (int K : {f.qk, 3 * f.qk, 1024, 5120, 17408})
            for (int N : {1, 5, 128, 129, 300, 5120, 17408})
                for (int M : {1, 2, 15, 16, 17, 100, 255, 256, 257, 512, 1000, 2048})
                    for (int sms : {152, 148, 132}) {
                        check_plan(fmt, N, K, M, sms);
                        ++plans;
                    }
    }
    printf("plans %ld fails %d\n", plans, fails);
    return fails ? 1 : 0;
}
