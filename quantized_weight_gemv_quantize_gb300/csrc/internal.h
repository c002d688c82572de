// Host-side declarations shared by the libqgemv translation units (not part of the public ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace qg {

// Kernel arguments of the staged GEMV kernels (all formats and the W8A16 variant).
struct GemvArgs {
    const uint8_t* W;       // weight stream, 16-byte aligned
    const uint8_t* x;       // q8_1 blocks, or bf16 activations for W8A16
    float* y;               // [m, N] fp32
    long long row_bytes;    // bytes of one weight row
    long long total_bytes;  // N * row_bytes
    int N, K;
    int rows_per_tile;      // rows per warp work item (R)
    int num_tiles;          // warp work items: ceil(N / R)
    int chunks;             // bulk copies per work item: 1 (R whole rows) or ceil(nb / chunk_blocks) (R == 1)
    int chunk_blocks;       // blocks per copy when a row is split (nb when chunks == 1)
    int blocks_per_row;     // nb
    int units_per_row;      // work units per row (see the kernel for the unit of each format)
    int lanes_log2;         // lanes per row team = 1 << lanes_log2 (<= 5)
    int stages;             // ring depth (<= MAX_STAGES)
    unsigned stage_bytes;   // bytes per ring slot (multiple of 128)
    unsigned x_off;         // byte offset of the activation staging area in dynamic shared memory
    unsigned w_off;         // byte offset of ring slot 0
    unsigned* err;          // device error word
};

constexpr int MAX_STAGES = 8;
constexpr int GEMV_THREADS = 256;

// Variant index used by the kernel tables: 0 Q4_K, 1 Q6_K, 2 Q8_0, 3 W8A16.
enum Variant { V_Q4K = 0, V_Q6K = 1, V_Q80 = 2, V_W8A16 = 3 };

// Bytes of activation staging in shared memory for a variant at (m, K); multiple of 128.
unsigned x_stage_bytes(int variant, int m, int K);

// Kernel entry for (variant, m) as a host function pointer, for attribute / occupancy queries.
const void* gemv_kernel_ptr(int variant, int m);

// Launch the staged GEMV kernel.
cudaError_t launch_gemv(int variant, int m, const GemvArgs& a, int grid, int threads, unsigned smem, cudaStream_t s);

// Activation quantizer launch: x fp32 [m, K] -> q8_1 blocks.
cudaError_t launch_quantize(const float* x, int m, int K, uint8_t* xq, cudaStream_t s);

}  // namespace qg
