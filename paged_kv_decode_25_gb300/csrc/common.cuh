// Device helpers shared by the append and attention kernels: bf16 bit
// conversions, inline-PTX wrappers for mbarriers, TMA tensor copies,
// ldmatrix / movmatrix / mma.sync, and the bounded mbarrier wait.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mi.h"

namespace mi {

constexpr int kBlock = 16;               // tokens per KV block
constexpr long long kWaitLimitNs = 2000000000LL;  // 2 s bound on any mbarrier wait
// Waits for asynchronous work a kernel has itself issued (its copies landing,
// its MMAs finishing) before it releases shared or tensor memory use at
// least this bound, however short a test makes the launch's wait limit.
constexpr long long kDrainMinNs = 10000000LL;     // 10 ms

__host__ __device__ inline long long drain_limit(long long wait_ns) {
    return wait_ns > kDrainMinNs ? wait_ns : kDrainMinNs;
}

// Failure-detection test settings (mi_test_set_wait_limit,
// mi_test_withhold_copy), read on the host when a launch's parameters are
// built: the launch's wait limit, and whether its producer withholds one
// staged copy.
long long test_wait_limit_ns();
bool test_withhold_copy();

// ------------------------------------------------------------------ bf16 ---

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

// fp32 -> bf16 bits, round to nearest even; NaN -> quiet NaN with the sign kept.
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    const uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    const uint32_t r = u + 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(r >> 16);
}

// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// double -> bf16 bits with a single rounding (nearest, ties to even), working
// on the binary64 fields: keep 8 significant bits (fewer below 2^-126, where
// the bf16 quantum is fixed at 2^-133), round the dropped bits, rebias.
__device__ __forceinline__ uint16_t f64_to_bf16(double x) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(x);
    const uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    const unsigned long long a = u & 0x7FFFFFFFFFFFFFFFull;
    if (a > 0x7FF0000000000000ull) return (uint16_t)(sign | 0x7FC0u);   // NaN
    const int e = (int)(a >> 52);                                      // biased exponent
    if (e == 0) return sign;                                           // zero / double subnormal
    if (e == 0x7FF) return (uint16_t)(sign | 0x7F80u);                 // infinity
    const int E = e - 1023;
    const int Ec = E < -126 ? -126 : E;
    const int drop = 45 + (Ec - E);                 // dropped low bits of the 53-bit significand
    if (drop > 54) return sign;                     // below half the smallest subnormal
    const unsigned long long m = (a & 0x000FFFFFFFFFFFFFull) | 0x0010000000000000ull;
    unsigned long long q = m >> drop;
    const unsigned long long rem = m & ((1ull << drop) - 1ull);
    const unsigned long long half = 1ull << (drop - 1);
    if (rem > half || (rem == half && (q & 1ull))) ++q;
    unsigned long long bits = ((unsigned long long)(Ec + 126) << 7) + q;
    if (bits >= 0x7F80ull) bits = 0x7F80ull;        // overflow -> infinity
    return (uint16_t)(sign | (uint16_t)bits);
}

// 2^x on the special-function unit (results below 2^-126 flush to zero,
// which for attention weights relative to the row max is immaterial).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------- errors ------

__device__ __forceinline__ void raise_err(int32_t* dev_err, int bit) {
    if (dev_err) atomicOr(dev_err, bit);
}

// -------------------------------------------------------------- PTX --------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Raises the barrier's expected transaction bytes without arriving (the
// caller arrives later, after writes the waiters must see).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Like mbar_try_wait, with a suspend-time hint: a thread whose phase has not
// completed may sleep up to hint_ns before the call returns false, and
// wakes when the phase completes. A waiting warp then polls rarely and
// leaves its scheduler's issue slots to the warps that work (a warp issuing
// tensor-core MMAs among busy warps gets few of them).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

constexpr uint32_t kWaitSleepNs = 50000;  // longest sleep of one poll; the limit is checked between polls

// Wait for phase `parity` of the barrier to complete, for at most limit_ns
// (the launch's wait limit: kWaitLimitNs unless a test shortened it), plus
// one poll's sleep when sleep_ns > 0 (each poll may then sleep that long;
// with 0 the thread polls without a hint). Returns false when the limit ran
// out. Which is faster depends on the kernel: measured per kernel.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit_ns,
                                                  uint32_t sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (sleep_ns > 0) {
            if (mbar_try_wait_sleep(bar, parity, sleep_ns)) return true;
        } else {
            for (int i = 0; i < 64; ++i)
                if (mbar_try_wait(bar, parity)) return true;
        }
        if ((long long)(globaltimer() - t0) > limit_ns) return false;
    }
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 3-D and 4-D tiled TMA loads (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z,
                                            int w, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ fp8 ---

// Two e4m3 codes (low byte first) -> f16x2 (low half first). Exact: every
// e4m3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    const unsigned short h = (unsigned short)(two & 0xFFFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

// ----------------------------------------------------------------- int8 ---

// Two int8 codes -> f16x2 (low half first), exact. `u` holds four codes with
// their sign bits flipped (code + 128, offset binary); `sel` picks bytes 0-1
// (0x4140) or 2-3 (0x4342). Each byte goes under 0x64, giving the f16 value
// 1024 + (code + 128); subtracting 1152 leaves the code, an integer f16
// holds exactly.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t u, uint32_t sel) {
    const uint32_t x = __byte_perm(u, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64806480u));
    return r;
}

// The same pair without the subtraction: f16 values 1152 + code, exact. A
// caller that multiplies them on tensor cores takes 1152 times the other
// operand's sum back off the result.
__device__ __forceinline__ uint32_t i8x2_to_f16x2_biased(uint32_t u, uint32_t sel) {
    return __byte_perm(u, 0x64646464u, sel);
}

// Two fp32 -> e4m3 codes (lo in the low byte), nearest-even, saturating to
// +-448 for finite values out of range.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 -> packed f16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float f16_lo(uint32_t w) {
    float f;
    const unsigned short h = (unsigned short)(w & 0xFFFFu);
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}

__device__ __forceinline__ float f16_hi(uint32_t w) {
    float f;
    const unsigned short h = (unsigned short)(w >> 16);
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
}

// ----------------------------------------------- programmatic launch -------

// A kernel launched with launch_pdl may start while the previous kernel in
// the stream is still running; it calls pdl_wait() before touching memory
// that kernel may write, and pdl_trigger() to let the next kernel start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Args>
inline cudaError_t launch_pdl(void (*fn)(Args...), int grid, int block, int smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, args...);
}

}  // namespace mi
