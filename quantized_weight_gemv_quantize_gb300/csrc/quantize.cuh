// One q8_1 block per eight lanes: lane `part` of the group owns values 4 part .. 4 part + 3 of block `blk`.
// Every lane of the warp must call it (the amax and the code sum are xor-shuffle reductions inside the
// eight-lane group); lanes with valid == false take part in the shuffles and store nothing.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace qg {

// Four consecutive values of the input row as exact fp32 (16-bit kinds widen exactly).
template <int XK>
__device__ __forceinline__ float4 load4(const void* x, size_t i4) {
    if constexpr (XK == ACT_F32) {
        return reinterpret_cast<const float4*>(x)[i4];
    } else {
        const uint2 w = reinterpret_cast<const uint2*>(x)[i4];
        if constexpr (XK == ACT_BF16) {
            return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                               __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
        } else {
            return make_float4(h2f(w.x), h2f(w.x >> 16), h2f(w.y), h2f(w.y >> 16));
        }
    }
}

template <int XK>
__device__ __forceinline__ void quantize_block_part(const void* __restrict__ x, int blk, int part, bool valid,
                                                    uint8_t* __restrict__ xq) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) v = load4<XK>(x, static_cast<size_t>(blk) * 8 + part);
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float d32 = __fdiv_rn(amax, 127.0f);
    const int q0 = q8_1_code(v.x, d32), q1 = q8_1_code(v.y, d32), q2 = q8_1_code(v.z, d32), q3 = q8_1_code(v.w, d32);
    int sum = q0 + q1 + q2 + q3;
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    if (!valid) return;
    uint8_t* out = xq + static_cast<size_t>(blk) * 36;
    const uint32_t packed = (static_cast<uint32_t>(q0) & 0xFFu) | ((static_cast<uint32_t>(q1) & 0xFFu) << 8) |
                            ((static_cast<uint32_t>(q2) & 0xFFu) << 16) | ((static_cast<uint32_t>(q3) & 0xFFu) << 24);
    reinterpret_cast<uint32_t*>(out + 4)[part] = packed;
    if (part == 0) {
        const __half dh = __float2half_rn(d32);
        const float sp = __half2float(dh) * static_cast<float>(sum);  // exact product
        const __half sh = __float2half_rn(sp);
        reinterpret_cast<uint32_t*>(out)[0] =
            static_cast<uint32_t>(__half_as_ushort(dh)) | (static_cast<uint32_t>(__half_as_ushort(sh)) << 16);
    }
}

}  // namespace qg
