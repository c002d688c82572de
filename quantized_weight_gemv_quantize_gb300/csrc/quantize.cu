// Activation quantizer: fp32 [m, K] -> q8_1 blocks (36 B per 32 values), bit-exact with the definition
// in include/qgemv.h.  Eight lanes own one block (four values each, one 16-byte load); the block amax and
// the code sum are xor-shuffle reductions inside the 8-lane group.  The quantize-once-per-input placement
// follows vllm.cpp PR #1936 (SGLang/vLLM study section), and the cooperative per-block layout follows its
// QuantizeQ8KKWarpCoop section (several lanes per block, shuffle amax).
#include "quantize.cuh"

namespace qg {

#ifdef QGEMV_TRACE
#define QG_TRACE_PARAM , unsigned long long* trace
#define QG_TRACE_ARG , trace
#else
#define QG_TRACE_PARAM
#define QG_TRACE_ARG
#endif

template <int XK>
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const void* __restrict__ x, int nblocks,
                                                            uint8_t* __restrict__ xq, int late QG_TRACE_PARAM) {
#ifdef QGEMV_TRACE
    const unsigned long long t_entry = global_ns();
#endif
    // Under programmatic dependent launch: let the next kernel start launching (at once, or with `late`
    // only after the wait) and wait for the producer of x (all no-ops otherwise).
    if (!late) pdl_launch_dependents();
    pdl_wait();
    if (late) pdl_launch_dependents();
#ifdef QGEMV_TRACE
    unsigned long long* tr =
        trace && blockIdx.x < TRACE_CTAS ? trace + static_cast<size_t>(blockIdx.x) * TRACE_FIELDS : nullptr;
    if (tr && threadIdx.x == 0) {
        tr[0] = t_entry;
        tr[1] = global_ns();
        tr[7] = 2;
    }
#endif
    const int gt = blockIdx.x * blockDim.x + threadIdx.x;
    const int blk = gt >> 3, part = gt & 7;
    quantize_block_part<XK>(x, blk, part, blk < nblocks, xq);
#ifdef QGEMV_TRACE
    __syncthreads();
    if (tr && threadIdx.x == 0) tr[2] = tr[3] = global_ns();
#endif
}

cudaError_t launch_quantize(int x_kind, const void* x, int m, int K, uint8_t* xq, bool pdl, bool late, cudaStream_t s) {
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
#ifdef QGEMV_TRACE
    unsigned long long* trace = trace_next_launch();
#endif
    cudaError_t e;
    const int lt = late ? 1 : 0;
    if (x_kind == ACT_BF16) e = cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<ACT_BF16>, x, nblocks, xq, lt QG_TRACE_ARG);
    else if (x_kind == ACT_F16) e = cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<ACT_F16>, x, nblocks, xq, lt QG_TRACE_ARG);
    else e = cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<ACT_F32>, x, nblocks, xq, lt QG_TRACE_ARG);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

}  // namespace qg
