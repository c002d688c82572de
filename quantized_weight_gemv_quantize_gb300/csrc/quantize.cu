// Activation quantizer: fp32 [m, K] -> q8_1 blocks (36 B per 32 values), bit-exact with the definition
// in include/qgemv.h.  Eight lanes own one block (four values each, one 16-byte load); the block amax and
// the code sum are xor-shuffle reductions inside the 8-lane group.  The quantize-once-per-input placement
// follows vllm.cpp PR #1936 (SGLang/vLLM study section), and the cooperative per-block layout follows its
// QuantizeQ8KKWarpCoop section (several lanes per block, shuffle amax).
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
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const void* __restrict__ x, int nblocks,
                                                            uint8_t* __restrict__ xq) {
    // Under programmatic dependent launch: let the next kernel start launching, then wait for the
    // producer of x (both no-ops otherwise).
    pdl_launch_dependents();
    pdl_wait();
    const int gt = blockIdx.x * blockDim.x + threadIdx.x;
    const int blk = gt >> 3, part = gt & 7;
    const bool valid = blk < nblocks;
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

cudaError_t launch_quantize(int x_kind, const void* x, int m, int K, uint8_t* xq, bool pdl, cudaStream_t s) {
    const int nblocks = m * (K / 32);
    const int threads = 256;
    const int grid = (nblocks * 8 + threads - 1) / threads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e;
    if (x_kind == ACT_BF16) e = cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<ACT_BF16>, x, nblocks, xq);
    else if (x_kind == ACT_F16) e = cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<ACT_F16>, x, nblocks, xq);
    else e = cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<ACT_F32>, x, nblocks, xq);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

}  // namespace qg
