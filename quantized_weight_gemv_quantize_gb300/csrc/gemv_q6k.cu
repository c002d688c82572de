// Instantiations of the staged GEMV kernel for one variant: kind 1..8 = m rows, kind 0 = the single-row
// streaming build, kind 9 = the single-row streaming build with the fused argmax,
// kind 10 = the 16-row build for m = 9..16, kinds 11 / 12 = the K-chunk builds of 8 / 16 rows, kind 13 = the
// 8-row build with row pairs.
#include "gemv_kernel.cuh"

namespace qg {

const void* gemv_kernel_ptr_q6k(int kind) {
    switch (kind) {
    case 0: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 1, true>);
    case 9: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 1, true, true>);
    case 1: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 1>);
    case 2: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 2>);
    case 3: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 3>);
    case 4: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 4>);
    case 5: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 5>);
    case 6: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 6>);
    case 7: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 7>);
    case 8: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 8>);
    case KIND_M16: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 16>);
    case KIND_M8_CHUNK: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 8, false, false, true>);
    case KIND_M16_CHUNK: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 16, false, false, true>);
    case KIND_M8_PAIR: return reinterpret_cast<const void*>(&gemv_staged_kernel<V_Q6K, 8, false, false, false, true>);
    }
    return nullptr;
}

}  // namespace qg
