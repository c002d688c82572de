// Device helpers shared by the libqgemv kernels (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qgemv.h"

namespace qg {

// Bits of the device-side error word.
enum : unsigned { ERR_WAIT_TIMEOUT = 1u, ERR_DRAIN_TIMEOUT = 2u };

// Upper bound on any on-chip wait, in ns of %globaltimer.  In a correct run a wait ends in microseconds;
// the bound only exists so that a broken wait can never hang the GPU.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Test the phase; the thread may sleep up to the suspend-time hint (ns) inside the instruction, so a
// waiting warp costs few issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the mbarrier; gives up after WAIT_LIMIT_NS and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
#pragma unroll 1
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
    return true;
}

// L2 policy for a stream read exactly once: evict first, so the weights do not push the (re-used)
// activations and outputs out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared (async proxy), completion counted on the mbarrier in bytes.
// dst, src 16-byte aligned; bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream start launching, and wait until the
// previous kernel's memory operations are visible.  Both are no-ops when the launch has no programmatic
// dependency.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// NW consecutive little-endian 32-bit words starting at a 2-byte aligned shared-memory address:
// aligned loads plus a funnel shift (shift 0 when the address is already 4-byte aligned).  Reads at
// most 4 bytes past the last requested byte.
template <int NW>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t (&w)[NW]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* base = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    uint32_t t[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) t[i] = base[i];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

// The same from an already aligned base and a known shift (8 x the address mod 4).
template <int NW>
__device__ __forceinline__ void lds_words_at(const uint32_t* base, uint32_t sh, uint32_t (&w)[NW]) {
    uint32_t t[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) t[i] = base[i];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

// q8_1 code of one value given the block's fp32 scale d32 = amax / 127: IEEE division, halfway cases away
// from zero, clamp to +-127; 0 when d32 == 0.  Shared by the standalone quantizer and the GEMV kernels'
// in-kernel quantization so both produce the same codes.
__device__ __forceinline__ int q8_1_code(float v, float d32) {
    if (d32 == 0.0f) return 0;
    float r = roundf(__fdiv_rn(v, d32));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

// Exact int -> float for |v| < 2^22 without the (quarter-rate) conversion unit: 0x4B400000 is 1.5 * 2^23,
// so the integer lands in the mantissa of a float whose spacing is 1; subtracting the bias is exact.
__device__ __forceinline__ float i2f_small(int v) {
    return __int_as_float(0x4B400000 + v) - 12582912.0f;
}

// A dp4a chain seeded with I2F_SEED ends at 0x4B400000 + s: for |s| < 2^22 the bits of the float 2^23 + 2^22 + s,
// so seeded_to_f32 gives s exactly with one add fewer than i2f_small.
constexpr int I2F_SEED = 0x4B400000;
__device__ __forceinline__ float seeded_to_f32(int v) { return __int_as_float(v) - 12582912.0f; }

// int8 byte j of v (v already xor 0x80808080, i.e. q + 128 unsigned) -> exact fp32 q:
// 0x4B0000uu is 2^23 + u as a float; subtracting 2^23 + 128 is exact.
__device__ __forceinline__ float s8_to_f32(uint32_t v_biased, int j) {
    return __uint_as_float(__byte_perm(v_biased, 0x4B000000u, 0x7650u | static_cast<unsigned>(j))) - 8388736.0f;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Four-way byte dot product with UNSIGNED bytes in a and signed bytes in b, accumulated into c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

}  // namespace qg
