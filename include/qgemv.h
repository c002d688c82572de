/*
 * libqgemv -- quantized-weight decode GEMV for NVIDIA GB300 (sm_103a), C ABI.
 *
 * The operation (vllm.cpp PR #1936 "raise Qwen3.5-4B Q4_K_M gfx1100 decode", the SGLang/vLLM study
 * section): for single-token decode, each activation row is quantized ONCE to q8_1-style int8 blocks,
 * then every output row streams its 4/6/8-bit super-blocks, dequantizes them in registers and reduces
 * the dot product:
 *
 *     y[i, n] = sum_k  w[n, k] * xhat[i, k]          i < m (1..16), n < N, k < K
 *
 * where w is the dequantized weight and xhat = d * q the dequantized activation.  The integer block dots
 * are exact; scales and the final reduction run in fp32.  The W8A16 entry (MetaInfer-cpp README, the
 * W8A16 section; zLLM article "Decode 只有一行", the W8/W8A16 direct-read section) multiplies int8
 * weights directly against 16-bit activations with fp32 accumulation, with no activation quantization.
 *
 * Block formats.  No page fixes a bit packing; these layouts are this library's own.  All multi-byte
 * fields are little-endian; fp16 is IEEE binary16; bf16 is the top half of an IEEE binary32.
 *
 *   q8_1 activation block (36 B per 32 values):
 *       [0..1]  d  fp16     scale; xhat = d * q
 *       [2..3]  s  fp16     binary16(float(d) * sum(q))   (informational; the GEMV never reads it)
 *       [4..35] qs int8[32] q[j] is value 32*b + j of the row
 *     A row of K values is K/32 consecutive blocks; row i starts at byte i * (K/32) * 36.
 *
 *   QGEMV_Q4_K super-block (144 B per 256 weights):
 *       [0..1]   d     fp16
 *       [2..3]   dmin  fp16
 *       [4..15]  a 96-bit little-endian bit string; field f (f = 0..15) is bits 6f..6f+5;
 *                fields 0..7 are sc[0..7], fields 8..15 are mn[0..7] (unsigned 6-bit)
 *       [16..143] qs[128]: byte 32g+t (g < 4, t < 32) holds code of element 64g+t in its low nibble and
 *                of element 64g+32+t in its high nibble
 *       w[e] = d * sc[e/32] * q[e] - dmin * mn[e/32]
 *
 *   QGEMV_Q6_K super-block (210 B per 256 weights):
 *       [0..127]   ql: byte 64h+t (h < 2, t < 64) holds the low 4 bits of element 128h+t (low nibble)
 *                  and of element 128h+64+t (high nibble)
 *       [128..191] qh: byte 32h+t (h < 2, t < 32) holds bits 4..5 of element 128h+32k+t in its bits
 *                  2k..2k+1 (k < 4)
 *       [192..207] sc int8[16]
 *       [208..209] d fp16
 *       w[e] = d * sc[e/16] * (q[e] - 32),  q[e] in 0..63
 *
 *   QGEMV_Q8_0 block (34 B per 32 weights):
 *       [0..1] d fp16, [2..33] qs int8[32];  w = d * q  (q may be -128..127)
 *
 *   QGEMV_Q5_K super-block (176 B per 256 weights; vllm.cpp PR #1936 decodes Q5_K in the same dp4a
 *   inner loops as Q4_K and Q6_K, the amd_mixed_dot section, and keeps its attention qkv tensors
 *   [2560 -> 8192] in Q5_K, the keep-quant section):
 *       [0..15]   d, dmin and the 96-bit sc/mn bit string, exactly as QGEMV_Q4_K
 *       [16..47]  qh[32]: bit j (j < 8) of byte t (t < 32) is bit 4 of element 32j+t
 *       [48..175] qs[128]: the low 4 bits of each element, packed as QGEMV_Q4_K's qs
 *       w[e] = d * sc[e/32] * q[e] - dmin * mn[e/32],  q[e] in 0..31
 *
 *   A weight matrix [N, K] is row-major: row n is K/256 (K-quants) or K/32 (Q8_0) consecutive blocks;
 *   rows are contiguous with no padding (row n starts at byte n * qgemv_weight_bytes(fmt, 1, K)).
 *
 * Common rules for every entry point:
 *   - All data pointers are caller-owned DEVICE memory.  The library never allocates, frees or keeps a
 *     pointer after the call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only enqueue work: they do
 *     not synchronize, and results are valid in stream order.
 *   - Argument errors are detected on the host before anything is enqueued; on any non-zero status
 *     nothing was launched and no output byte was written.
 *   - m (activation rows) is 1..16; larger m returns QGEMV_ERR_UNSUPPORTED (never a partial result).
 *     m = 1..8 run kernels built for that m.  m = 9..16 run one 16-row build (rows past m are staged
 *     as zeros and not stored), or, where K exceeds that build's activation staging, two launches of 8
 *     and m - 8 rows; each output row gets the same arithmetic either way.
 *   - K is at most qgemv_max_k (131072 at every m).  A launch stages the whole activation row in shared
 *     memory; rows longer than one pass of staging at the call's m (qgemv_chunk_k(fmt, m, K) < K) run as
 *     one launch per K-chunk: each launch reads only its chunk of every weight row (every weight byte is
 *     still read once), stages only its chunk of the activation, and every launch after the first adds
 *     its partial sums to y, in stream order (no atomics; the result does not depend on timing).  A
 *     row's summation order is then fixed by (fmt, K, m) rather than (fmt, K).
 *   - Outputs are fully overwritten (no accumulation into y).
 *   - Inputs must be finite; a NaN or Inf in x gives unspecified output (no trap, no fault).
 *   - Thread safety: calls may be made from several host threads on different streams.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>

#if defined(__GNUC__)
#define QGEMV_API __attribute__((visibility("default")))
#else
#define QGEMV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QGEMV_Q4_K = 1,
    QGEMV_Q6_K = 2,
    QGEMV_Q8_0 = 3,
    QGEMV_W8A16 = 4, /* Q8_0 weights against bf16 activations (qgemv_multi only; see qgemv_w8a16) */
    QGEMV_Q5_K = 5,
    QGEMV_W8A16_CHANNEL = 6 /* per-channel INT8 weights against bf16 activations (qgemv_plan_info only) */
} qgemv_fmt;

/* Activation kinds for qgemv_multi. */
typedef enum {
    QGEMV_ACT_Q8_1 = 0, /* q8_1 blocks as written by qgemv_quantize_act                       */
    QGEMV_ACT_F32 = 1,  /* fp32 [m, K]: quantized inside the GEMV launch (same bits as the quantizer) */
    QGEMV_ACT_BF16 = 2, /* bf16 [m, K]: W8A16 (not quantized), or qgemv_quantize_act_typed input   */
    QGEMV_ACT_F16 = 3   /* IEEE binary16 [m, K]: qgemv_quantize_act_typed input                    */
} qgemv_act;

/*
 * Launch flags (the *_ex and qgemv_multi entry points).
 *
 * QGEMV_FLAG_PDL: launch with programmatic dependent launch (sm_90+ stream semantics).  The kernel may
 * start while the kernels before it in the stream are still running, and it starts streaming its first
 * weight tiles from that moment; it waits for those kernels before it reads the activation or writes any
 * output.  The caller guarantees that the weight buffers are not written by kernels still in flight when
 * the call is enqueued.  Under CUDA graphs this removes most of the gap between consecutive decode
 * kernels.
 *
 * QGEMV_FLAG_PDL_LATE_TRIGGER (the quantizer entry points only, with QGEMV_FLAG_PDL): the launch lets the
 * next kernel of the stream start only once its own wait for the kernels before it has ended, instead of
 * at once.  It is a scheduling hint and changes no result.  Measured: before a short GEMV (weights below
 * about 4 MB, the launches of the register-capped single-row build) the later start was faster, the
 * following short launches above all; before a long GEMV it was slower, because that GEMV's weights
 * start streaming later.
 */
#define QGEMV_FLAG_PDL 1u
#define QGEMV_FLAG_PDL_LATE_TRIGGER 2u

/* Up to this many matrices share one activation in one qgemv_multi launch. */
#define QGEMV_MAX_GROUP 8

/* One weight matrix of a qgemv_multi group: W in the group's format, y fp32 [m, N]. */
typedef struct {
    const void* W;
    float* y;
    int N;
} qgemv_mat;

typedef enum {
    QGEMV_OK = 0,
    QGEMV_ERR_INVALID_ARG = 1, /* null pointer, bad format, non-positive size, K not a block multiple */
    QGEMV_ERR_UNSUPPORTED = 2, /* valid but outside the library's limits (m > 16, K too large for m)  */
    QGEMV_ERR_MISALIGNED = 3,  /* a pointer violates its alignment rule                              */
    QGEMV_ERR_CUDA = 4,        /* the CUDA runtime reported an error (see qgemv_last_cuda_error)      */
    QGEMV_ERR_DEVICE = 5,      /* the current device is not a compute-capability 10.3 (GB300) part    */
    QGEMV_ERR_OVERLAP = 6      /* the output range overlaps an input range                            */
} qgemv_status;

/*
 * Activation quantizer: x fp32 [m, K] row-major  ->  xq, m * (K/32) q8_1 blocks (qgemv_act_bytes(m, K)).
 *
 * Per block of 32 values (vllm.cpp PR #1936, QuantizeQ8KK / warp-coop section: block amax, scale
 * amax/127, nearest integer, clamp to 127; SGLang/vLLM study section: q8_1 = 32 int8 + scale + sum):
 *     amax = max|x|;  d32 = amax / 127 (fp32 IEEE division);  d = binary16_rne(d32);
 *     q = clamp(roundf(x / d32), -127, 127)   (IEEE fp32 division, halfway cases away from zero;
 *                                              q = 0 everywhere when d32 == 0);
 *     s = binary16_rne(float(d) * sum(q))     (the fp32 product is exact).
 * Codes and both fp16 fields are bit-exact with that definition.
 *
 * x: 16-byte aligned, m*K floats.  xq: 16-byte aligned, qgemv_act_bytes(m, K) bytes, not overlapping x.
 * 1 <= m <= 16, K > 0, K % 32 == 0.
 */
QGEMV_API int qgemv_quantize_act(const float* x, int m, int K, void* xq, void* stream);

/*
 * Quantized GEMV: y[i, n] = sum_k w[n, k] * xhat[i, k]   (fp32 out, [m, N] row-major).
 *
 * W: 16-byte aligned, qgemv_weight_bytes(fmt, N, K) bytes in the `fmt` layout above.
 * xq: 16-byte aligned, m*(K/32) q8_1 blocks as written by qgemv_quantize_act (row i = activation row i).
 * y: 4-byte aligned, m*N floats, must not overlap W or xq.
 * 1 <= m <= 16, N >= 1, K % 256 == 0 for Q4_K/Q5_K/Q6_K, K % 32 == 0 for Q8_0, K <= qgemv_max_k(fmt, m).
 * Integer block dots are exact; per-block scaling and the reduction are fp32, so y matches the exact
 * value to fp32 rounding (relative L2 error well under 1e-5 on N(0,1) activations).
 * Each output row's result depends only on its own weight row and the activation: stacking two weight
 * matrices row-wise concatenates their outputs bit for bit.
 */
QGEMV_API int qgemv(int fmt, const void* W, const void* xq, float* y, int m, int N, int K, void* stream);

/*
 * W8A16: y[i, n] = sum_b d[n, b] * sum_{j<32} q[n, 32b+j] * x[i, 32b+j]   (fp32 accumulation)
 *
 * W: Q8_0 layout, 16-byte aligned.  x_bf16: bf16 [m, K] row-major, 16-byte aligned.  y: fp32 [m, N],
 * 4-byte aligned, not overlapping W or x.  1 <= m <= 16, K % 32 == 0, K <= qgemv_max_k_w8a16(m).
 */
QGEMV_API int qgemv_w8a16(const void* W, const void* x_bf16, float* y, int m, int N, int K, void* stream);

/*
 * The activation quantizer for 16-bit activation rows: x_kind QGEMV_ACT_BF16 or QGEMV_ACT_F16 (or
 * QGEMV_ACT_F32, the same as qgemv_quantize_act).  Every 16-bit value widens exactly to fp32, and the q8_1
 * definition above is then applied unchanged, so the blocks are bit-identical to qgemv_quantize_act on
 * the widened rows.  (vllm.cpp PR #1936 quantizes the engine's activations, which its engines keep in
 * 16-bit types, the SGLang/vLLM study section; the library's own addition.)
 * x: 16-byte aligned, m*K values of the given kind; other rules as qgemv_quantize_act.  flags: 0,
 * QGEMV_FLAG_PDL, or QGEMV_FLAG_PDL | QGEMV_FLAG_PDL_LATE_TRIGGER (any other bit: QGEMV_ERR_INVALID_ARG).
 */
QGEMV_API int qgemv_quantize_act_typed(int x_kind, const void* x, int m, int K, void* xq, unsigned flags,
                                       void* stream);

/*
 * Per-output-channel INT8 W8A16 (MetaInfer-cpp README, the Qwen3-14B TP4 W8A16 decode section: signed
 * INT8 weights, one fp32 scale per output channel, bf16 activations, fp32 accumulation):
 *     y[i, n] = scale[n] * sum_k Wq[n, k] * x[i, k]
 * The sum is accumulated in fp32 over the exact products and multiplied by scale[n] once.
 * Wq: int8 [N, K] row-major (any value -128..127; symmetric quantizers write -127..127), 16-byte aligned.
 * scale: fp32 [N], 4-byte aligned.  x_bf16: bf16 [m, K], 16-byte aligned.  y: fp32 [m, N], 4-byte aligned,
 * not overlapping the inputs.  1 <= m <= 16, K % 32 == 0, K <= qgemv_max_k_w8a16_channel(m).
 */
QGEMV_API int qgemv_w8a16_channel(const void* Wq, const float* scale, const void* x_bf16, float* y, int m, int N,
                                  int K, void* stream);
QGEMV_API int qgemv_w8a16_channel_ex(const void* Wq, const float* scale, const void* x_bf16, float* y, int m,
                                     int N, int K, unsigned flags, void* stream);
QGEMV_API int qgemv_max_k_w8a16_channel(int m);

/*
 * GEMV with a fused argmax (the lm_head of greedy decoding): y = W * xhat as qgemv computes it, but y is
 * not written; idx_out[i] receives the first n with the largest y[i, n], val_out[i] that y value (NaN
 * counts as larger than every number, as in torch.argmax: a row whose y holds NaN gives the first NaN's
 * n; y itself can only hold NaN when an input is not finite).  Each CTA
 * reduces its rows, and the last CTA to finish combines the CTAs' results, so one launch replaces the
 * GEMV and a separate argmax pass.  (MetaInfer-cpp README, the device-sampling section: an lm_head that
 * returns the argmax without writing the logits; vllm.cpp PR #1936, the split-argmax section: ties go to
 * the lower index, which makes the combine associative and the result independent of its order.)
 * fmt: QGEMV_Q4_K / QGEMV_Q5_K / QGEMV_Q6_K / QGEMV_Q8_0, q8_1 activations, m = 1 (other m return
 * QGEMV_ERR_UNSUPPORTED).
 * scratch: device memory of at least qgemv_argmax_scratch_bytes(m) bytes, 16-byte aligned, whose first
 * 4 bytes must be zero before the first call (e.g. cudaMemset once); each call leaves them zero again.
 * Calls that share one scratch buffer must be ordered (same stream, or synchronized): concurrent calls
 * on the same scratch race.  idx_out: int[m], val_out: float[m], 4-byte aligned, not overlapping the
 * inputs or the scratch.
 */
QGEMV_API size_t qgemv_argmax_scratch_bytes(int m);
QGEMV_API int qgemv_argmax(int fmt, const void* W, const void* xq, int m, int N, int K, void* scratch,
                           size_t scratch_bytes, int* idx_out, float* val_out, unsigned flags, void* stream);

/*
 * qgemv_argmax on a scratch the library owns, for callers that have no allocator at hand.  The pages have
 * no counterpart of this entry point; it adds no arithmetic of its own.
 * The scratch is a fixed array of QGEMV_ARGMAX_STATIC_SCRATCH_BYTES bytes in the library's static device
 * memory, one per device.  A call allocates nothing (no cudaMalloc, no allocating library call).
 * - Size limit: a call that would need more than QGEMV_ARGMAX_STATIC_SCRATCH_BYTES of scratch
 *   (qgemv_argmax_scratch_bytes(m) > the limit, i.e. m >= 2) returns QGEMV_ERR_UNSUPPORTED before touching
 *   the device; m outside 1..8 returns QGEMV_ERR_INVALID_ARG.
 * - Zero at start: the array's first 4 bytes (the CTAs' arrival counter) must be zero when a call starts.
 *   Static device memory is zero when the library's module is loaded on a device, and every call that runs
 *   to completion leaves the counter at zero again; the rest of the array needs no initial value.
 * - Setup: the first call on each device looks up the array's device address (cudaGetSymbolAddress) and
 *   does qgemv_argmax's own first-call setup.  That first call must happen before any stream capture.
 * - Races: every call on a device shares the one array.  Calls must be ordered (one stream, or
 *   synchronized); calls that overlap in time, on different streams or from different threads, race on
 *   the counter and the partial results, and their outputs are undefined.
 * Otherwise the arguments, validation and results are those of qgemv_argmax.
 */
#define QGEMV_ARGMAX_STATIC_SCRATCH_BYTES 16384
QGEMV_API int qgemv_argmax_noalloc(int fmt, const void* W, const void* xq, int m, int N, int K, int* idx_out,
                                   float* val_out, unsigned flags, void* stream);

/* As qgemv_quantize_act / qgemv / qgemv_w8a16, with launch flags (QGEMV_FLAG_PDL or 0; the quantizer also
 * takes QGEMV_FLAG_PDL_LATE_TRIGGER, which the GEMV entry points reject with QGEMV_ERR_INVALID_ARG). */
QGEMV_API int qgemv_quantize_act_ex(const float* x, int m, int K, void* xq, unsigned flags, void* stream);
QGEMV_API int qgemv_ex(int fmt, const void* W, const void* xq, float* y, int m, int N, int K, unsigned flags,
                       void* stream);
QGEMV_API int qgemv_w8a16_ex(const void* W, const void* x_bf16, float* y, int m, int N, int K, unsigned flags,
                             void* stream);

/*
 * Several matrices that read the same activation, in one launch: y_j = W_j xhat for j < count
 * (e.g. the q/k/v or gate/up projections of a layer, as vllm.cpp PR #1936's merged gate+up section does
 * by stacking rows; here the matrices stay separate buffers).  Every output equals what the
 * single-matrix call returns, bit for bit (each row's result depends only on its own weights and the
 * activation).
 *
 * fmt: QGEMV_Q4_K / QGEMV_Q5_K / QGEMV_Q6_K / QGEMV_Q8_0 with act_kind QGEMV_ACT_Q8_1 or QGEMV_ACT_F32, or
 *      QGEMV_W8A16 with act_kind QGEMV_ACT_BF16.
 * act: the shared activation (16-byte aligned): q8_1 blocks, fp32 [m, K] or bf16 [m, K].
 *      With QGEMV_ACT_F32 the launch quantizes the rows itself (the quantizer folded into the GEMV, so
 *      one fewer launch per input); the codes are bit-identical to qgemv_quantize_act's.
 * xq_out: QGEMV_ACT_F32 only; if not NULL the launch also writes the q8_1 blocks there (16-byte aligned,
 *      qgemv_act_bytes(m, K) bytes) for later calls on the same input.  Must be NULL otherwise.
 * 1 <= count <= QGEMV_MAX_GROUP; every W_j 16-byte aligned in `fmt`; every y_j 4-byte aligned; no output
 * overlaps another output or any input.  Same limits on m and K as qgemv.
 */
QGEMV_API int qgemv_multi(int fmt, int count, const qgemv_mat* mats, int act_kind, const void* act, void* xq_out,
                          int m, int K, unsigned flags, void* stream);

/* Sizes in bytes; 0 for an invalid (fmt, N, K) or (m, K). */
QGEMV_API size_t qgemv_weight_bytes(int fmt, int N, int K);
QGEMV_API size_t qgemv_act_bytes(int m, int K);

/* Largest K the library serves at a given m (131072; rows beyond one pass of activation staging run as
 * K-chunks); 0 for an invalid argument. */
QGEMV_API int qgemv_max_k(int fmt, int m);
QGEMV_API int qgemv_max_k_w8a16(int m);

/*
 * Values per K-chunk of a call at (fmt, m, K): K itself when the rows take one pass of activation staging,
 * else the chunk width (a multiple of 256; every chunk that wide but the last).  fmt may also be
 * QGEMV_W8A16 or QGEMV_W8A16_CHANNEL.  0 for an invalid argument or K beyond qgemv_max_k.  The fused
 * argmax needs one pass (qgemv_chunk_k(fmt, 1, K) == K).  No device needed.
 */
QGEMV_API int qgemv_chunk_k(int fmt, int m, int K);

/* Human-readable status name (static string; never NULL). */
QGEMV_API const char* qgemv_status_string(int status);

/* The cudaError_t value behind the most recent QGEMV_ERR_CUDA on the calling thread (0 if none). */
QGEMV_API int qgemv_last_cuda_error(void);

/*
 * Route counters: how many times each kernel variant was launched by this process (a witness of which
 * path ran).  Fills out[0 .. min(n, QGEMV_NUM_ROUTES)-1] and returns QGEMV_NUM_ROUTES.
 * Route ids: 0 quantizer, 1..8 Q4_K at m=1..8, 9..16 Q6_K, 17..24 Q8_0, 25..32 W8A16, 36..43 Q5_K,
 * 44..51 per-channel INT8 W8A16 (one count per GEMV launch at m <= 8); 53 launches of the 16-row build
 * (m = 9..16, any format); 52 launches with the fused argmax; 33 launches that quantized fp32
 * activations in-kernel, 34 launches over >= 2 matrices, 35 launches with programmatic dependent launch
 * (quantizer included), 54 launches that covered one K-chunk of long rows.
 */
#define QGEMV_ROUTE_FUSED 33
#define QGEMV_ROUTE_GROUPED 34
#define QGEMV_ROUTE_PDL 35
#define QGEMV_ROUTE_Q5_K_M1 36
#define QGEMV_ROUTE_W8A16_CHANNEL_M1 44
#define QGEMV_ROUTE_ARGMAX 52
#define QGEMV_ROUTE_M16 53 /* a launch of the 16-row build (m = 9..16), any format */
#define QGEMV_ROUTE_CHUNKED 54 /* a launch that covered one K-chunk of the rows (also counted by format) */
#define QGEMV_NUM_ROUTES 55
QGEMV_API int qgemv_route_counts(unsigned long long* out, int n);
QGEMV_API void qgemv_route_reset(void);

/*
 * Launch-plan introspection (no device needed): the plan the GEMV would use for (fmt, m, N, K) on a part
 * with `num_sms` SMs and `ctas_per_sm` resident CTAs.  fmt = QGEMV_W8A16 (4) asks for the W8A16 kernel,
 * QGEMV_W8A16_CHANNEL (6) for the per-channel INT8 kernel.  Fills
 * out[0..12] = {lanes per row team, rows per tile, tiles, ring stages, bytes per ring slot, dynamic shared
 * memory bytes, grid, bytes per weight row, work units per row, activation staging bytes, threads per
 * CTA, warps per row team, multi-warp reduction bytes, kernel build (m for the m-row kernel, 0 for the
 * single-row streaming build)} (out must hold 14 values).  For K beyond one pass of staging, the plan of
 * the call's first K-chunk launch.
 */
QGEMV_API int qgemv_plan_info(int fmt, int m, int N, int K, int num_sms, int ctas_per_sm, long long* out);

/*
 * The plan of one K-chunk launch covering Kc values of each of N rows (rows longer than one pass of
 * staging run as such launches; qgemv_chunk_k gives the chunk width, the last chunk may be narrower).
 * Fills out[0..14]: qgemv_plan_info's 14 values (row bytes are the chunk's), then the bytes from one row to
 * the next in a ring slot (each row's chunk arrives as its own copy).  Kc beyond one chunk launch's
 * staging returns QGEMV_ERR_UNSUPPORTED.  No device needed.
 */
QGEMV_API int qgemv_plan_info_chunk(int fmt, int m, int N, int Kc, int num_sms, int ctas_per_sm, long long* out);

/*
 * Tuning hook for sweeps: forces the resident CTAs per SM that the grid is sized for (1..4), log2 lanes
 * per row team (2..5), rows per tile, ring stages (2..8) and the single-row kernel build (1 = the
 * register-capped build for short launches, 2 = the streaming build) for every later GEMV launch in the
 * process; a value outside its range (e.g. 0 or -1) leaves that choice to the planner.  Not for
 * production use: forced plans are only checked for shared-memory fit.
 */
/* Tuning hook: row pairs (two rows per row team, for the builds that have them) 0 = planner decides,
 * 1 = whenever they fit, 2 = never.  Rows are bit-identical either way. */
QGEMV_API void qgemv_tune_pairs(int mode);

QGEMV_API void qgemv_tune_override(int ctas_per_sm, int lanes_log2, int rows_per_tile, int stages,
                                   int kernel_build);

/*
 * Failure injection for callers' error paths (host side only): the next `count` entry-point calls on
 * any thread return `status` without launching anything.  count = 0 disarms it.
 */
QGEMV_API void qgemv_debug_fail_next(int status, int count);

/*
 * Device-side error word.  Kernels never trap: a bounded on-chip wait that gives up (it cannot in a
 * correct run) sets a bit here and the kernel returns.  Reads (and with reset != 0 clears) the word for
 * the current device; this call synchronizes the device.  Returns a status.
 */
QGEMV_API int qgemv_device_error(unsigned int* out, int reset);

/*
 * Launch timeline (diagnostics).  A traced build of the library (libqgemv_trace.so, compiled with
 * QGEMV_TRACE) stamps %globaltimer at fixed points of every CTA of the first `launches` kernel launches
 * after qgemv_trace_begin, into a buffer in its static device memory; the normal build does no tracing
 * and these calls return QGEMV_ERR_UNSUPPORTED.  Launch numbers are assigned when a launch is enqueued
 * (under stream capture: when it is captured, so a replayed graph rewrites the same records).
 *   qgemv_trace_info:  the buffer's shape: launches x ctas records of `fields` unsigned 64-bit values.
 *   qgemv_trace_begin: zero the buffer and restart the numbering at 0 (synchronizes the device).
 *   qgemv_trace_read:  copy the first `bytes` of the buffer to host memory; *launches receives how many
 *                      launches have been numbered since qgemv_trace_begin (capped at the buffer's size).
 * Record of (launch, CTA): 0 kernel entry, 1 dependency released, 2 activation staged, 3 CTA done,
 * 4 producer issued its last tile, 5 producer's copies all landed, 6 SM id, 7 kind (1 GEMV, 2 quantizer),
 * 8..13 the first three tiles' (full-slot wait done, decode done) times of consumer warp 0; times in ns,
 * unused fields 0.  Timing only: a traced launch computes exactly what an untraced one does.
 */
QGEMV_API int qgemv_trace_info(int* launches, int* ctas, int* fields);
QGEMV_API int qgemv_trace_begin(void);
QGEMV_API int qgemv_trace_read(unsigned long long* host, size_t bytes, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
