// Host-side declarations shared by the libqgemv translation units (not part of the public ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace qg {

// Kernel arguments of the staged GEMV kernels (all formats and the W8A16 variant).
constexpr int MAX_GROUP = 8;  // matrices sharing one activation in one launch

// Activation kinds accepted by the GEMV kernels.
enum ActKind { ACT_Q8_1 = 0, ACT_F32 = 1, ACT_BF16 = 2, ACT_F16 = 3 };

struct GemvArgs {
    const uint8_t* W[MAX_GROUP];      // weight streams, 16-byte aligned
    float* y[MAX_GROUP];              // [m, N_j] fp32 outputs
    const float* rscale[MAX_GROUP];   // per-output-row fp32 scales [N_j] (per-channel INT8 only)
    long long total_bytes[MAX_GROUP]; // N_j * row_bytes
    int N[MAX_GROUP];
    int tile_start[MAX_GROUP + 1];    // first tile of matrix j; tile_start[count] = total tiles
    int count;                        // matrices in the group
    const uint8_t* x;       // q8_1 blocks (ACT_Q8_1), fp32 (ACT_F32) or bf16 (ACT_BF16) activations
    uint8_t* xq_out;        // ACT_F32 only: if not null, CTA 0 also writes the q8_1 blocks here
    int act;                // ActKind
    long long row_bytes;    // bytes of one weight row
    int K;
    int rows_per_tile;      // R: rows per tile (one bulk copy)
    int num_tiles;          // total tiles over the group
    int units_per_row;      // work units per row (see the kernel for the unit of each format)
    int lanes_log2;         // row team of 1 << lanes_log2 lanes (<= 32) when team_warps == 1
    int team_warps;         // G: warps per row team (1, or 2..8 for long rows)
    int stages;             // ring depth (<= MAX_STAGES)
    unsigned stage_bytes;   // bytes per ring slot (multiple of 128)
    unsigned red_off;       // byte offset of the multi-warp reduction area in dynamic shared memory
    unsigned x_off;         // byte offset of the activation staging area
    unsigned w_off;         // byte offset of ring slot 0
    unsigned* err;          // device error word
    // Fused argmax (single matrix): when am_scratch is set, rows are not written to y; instead
    // am_idx[i] / am_val[i] receive the first row n with the largest y[i, n].  am_scratch: an arrival
    // counter (4 bytes, zero before the launch and zero again after it) at offset 0, per-CTA partials
    // from offset 256.
    uint8_t* am_scratch;
    int* am_idx;
    float* am_val;
    int m_rows;             // activation rows of the call (the padded 16-row build serves m = 9..16)
    int row_pairs;          // builds with pair_rows(): 1 = teams decode two rows at once (tiles sized so)
    // K-chunked calls (rows longer than one pass of activation staging): each launch covers the values
    // [x_col_off, x_col_off + K) of every row; later chunks add their partial sums to y in stream order.
    long long w_row_stride;    // bytes from one weight row to the next in global memory (row_bytes unless chunked)
    long long w_col_off;       // byte offset of the chunk within each weight row
    unsigned slot_row_stride;  // 0: a tile's rows arrive as one contiguous copy; else one copy per row, at this
                               // stride (a multiple of 16) in the slot, each at its own 16-byte phase
    int x_row_stride;          // values from one activation row to the next (K unless chunked)
    int x_col_off;             // first activation value of the chunk (a multiple of 256)
    int accumulate;            // 1: add to y instead of writing it
#ifdef QGEMV_TRACE
    unsigned long long* trace;  // this launch's records (TRACE_CTAS x TRACE_FIELDS), or null
#endif
};

#ifdef QGEMV_TRACE
// Launch timeline of the traced build: one record of TRACE_FIELDS u64 per (launch, CTA) for the first
// TRACE_LAUNCHES launches after qgemv_trace_begin, CTAs below TRACE_CTAS.  Fields (ns of %globaltimer unless
// noted): 0 kernel entry, 1 dependency released (consumer side), 2 activation staged, 3 end of the CTA's work,
// 4 producer issued its last tile, 5 producer's copies all landed, 6 SM id, 7 kind (1 GEMV, 2 quantizer),
// 8/9, 10/11, 12/13: the first three tiles' full-barrier wait done / decode done (consumer warp 0).
constexpr int TRACE_LAUNCHES = 640, TRACE_CTAS = 320, TRACE_FIELDS = 16;
// Records of the next launch (advances the launch numbering); null past TRACE_LAUNCHES.
unsigned long long* trace_next_launch();
#endif

// Scratch of the fused argmax: the counter, then one (value, row) pair per CTA and activation row.
constexpr unsigned AM_SCRATCH_HEAD = 256;
constexpr unsigned AM_MAX_GRID = 1024;

constexpr int MAX_STAGES = 8;
constexpr int GEMV_CONSUMER_WARPS = 8;
constexpr int GEMV_THREADS_MAX = 32 * (GEMV_CONSUMER_WARPS + 1);
// Single-row kernels are compiled for four resident CTAs per SM (<= 56 registers): short launches then
// overlap, since up to four consecutive launches can each hold a CTA on an SM with its weights already
// in flight.
constexpr int GEMV_MIN_CTAS_M1 = 4;

// Variant index used by the kernel tables: 0 Q4_K, 1 Q6_K, 2 Q8_0, 3 W8A16, 4 Q5_K, 5 per-channel INT8
// weights against bf16 activations.
enum Variant { V_Q4K = 0, V_Q6K = 1, V_Q80 = 2, V_W8A16 = 3, V_Q5K = 4, V_W8C = 5 };
constexpr int NUM_VARIANTS = 6;

// Bytes of activation staging in shared memory for a variant at (m, K); multiple of 128.
unsigned x_stage_bytes(int variant, int m, int K);

// Kernel builds ("kinds"): 1..8 = the m-row kernel, 0 = the single-row streaming build, 9 = the single-row
// streaming build with the fused argmax, 10 = the 16-row build for m = 9..16 (rows past m padded),
// 11 / 12 = the K-chunk builds of 8 / 16 rows, 13 = the 8-row build with row pairs (pair_build).
constexpr int KIND_M16 = 10;
// K-chunk builds: 8 rows (m = 1..8, rows past m padded) and 16 rows (m = 9..16).
constexpr int KIND_M8_CHUNK = 11, KIND_M16_CHUNK = 12;
constexpr int KIND_M8_PAIR = 13;
constexpr int NUM_KINDS = 14;
constexpr int MAX_M = 16;

// Builds whose lane teams may decode two consecutive rows at once, each staged activation load serving
// both rows: Q4_K at m = 4..8 (these launches are bound by shared-memory load wavefronts).  Tiles then hold
// two rows per team.  Q6_K pairs rows at m = 8 in a build of its own (pair_build).  (Measured and left
// out: Q6_K at m = 4 and the single-row streaming builds of Q6_K and W8A16, where the larger tiles or the
// registers cost resident CTAs.)
__host__ __device__ constexpr bool pair_rows(int variant, int M) {
    return variant == V_Q4K && M >= 4 && M <= 8;
}

// Q6_K at m = 8 decodes row pairs in a build of its own (KIND_M8_PAIR): the pair path takes the 8-row
// build from 111 to 168 registers, which the launches without pairs (multi-warp teams, K = 9728) would pay
// too.  Measured: the 151936 x 2560 lm_head at m = 8 200.9 -> 152.5 us; with the pair path inside the
// common 8-row build the 4B-class m = 8 sweep was slower (2332.6 -> 2341.2 us).
__host__ __device__ constexpr bool pair_build(int variant, int M) {
    return variant == V_Q6K && M == 8;
}

// Kernel entry for (variant, kind) as a host function pointer, for attribute / occupancy queries.
const void* gemv_kernel_ptr(int variant, int kind);

// Launch the staged GEMV kernel (pdl: programmatic dependent launch attribute).
cudaError_t launch_gemv(int variant, int kind, const GemvArgs& a, int grid, int threads, unsigned smem, bool pdl,
                        cudaStream_t s);

// Activation quantizer launch: x fp32 [m, K] -> q8_1 blocks.
// Quantizer launch; x_kind is ACT_F32, ACT_BF16 or ACT_F16 (the input element type).
// late: the next kernel may start only after this one's own dependency wait (QGEMV_FLAG_PDL_LATE_TRIGGER).
cudaError_t launch_quantize(int x_kind, const void* x, int m, int K, uint8_t* xq, bool pdl, bool late, cudaStream_t s);

}  // namespace qg
