// Staged decode-GEMV kernel for the block-quantized formats (sm_103a).
//
// Data path, per CTA (persistent; the grid covers the SMs):
//   1. The activation (q8_1 blocks; fp32 rows, quantized by the CTA itself; or bf16 for W8A16) is staged
//      once into shared memory in a decode-friendly form: codes in bank-padded groups, fp32 block scales,
//      and per-format integer sums.
//   2. A producer warp streams tiles of whole weight rows (16-48 KB) into a ring of shared-memory slots
//      with one bulk copy per tile (cp.async.bulk, mbarrier completion, L2 evict-first).  Tiles that do
//      not start on a 16-byte boundary (Q6_K / Q8_0 rows) are copied as the aligned superset; the
//      decoder indexes from the remainder.
//   3. Consumer warps decode the rows of each tile in row teams; each work unit dequantizes its codes in
//      registers, forms exact int32 dots with dp4a against the staged activation codes, and applies the
//      fp32 block scales.  Partials are reduced with xor-shuffles (and, for rows split over several
//      warps, in shared memory in a fixed order).
//
// Work unit per format (64 weights for the K-quants, 32 for Q8_0):
//   Q4_K : one 32-byte slice g of qs -> sub-blocks 2g (low nibbles) and 2g+1 (high nibbles).
//   Q5_K : as Q4_K, with bits 2g and 2g+1 of the 32 qh bytes as bit 4 of the codes.
//   Q6_K : one half h of the block and 16 of its 32 qh columns -> 16 values in each of 4 sub-blocks.
//   Q8_0 : one block.
//   W8A16: one block (int8 weights times bf16 activations in fp32, no dp4a).
//   per-channel INT8: 32 consecutive weights (no block scale; the row's scale is applied at the store).
// Q4_K at m = 4..8 may decode two rows per team (row pairs): each staged activation load then serves
// both rows, and each row's arithmetic is the single-row unit's.
// This follows the "one warp per output row, dequantize in registers" decode of vllm.cpp PR #1936
// (the MMVQ geometry and T20 full-warp-cooperation sections), with the lanes per row made a plan
// parameter and the weight movement handed to the bulk-copy engine.
#pragma once
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace qg {

template <int V>
struct Traits;
template <>
struct Traits<V_Q4K> {
    static constexpr int BB = 144, BE = 256, UPB = 4;
};
template <>
struct Traits<V_Q5K> {
    static constexpr int BB = 176, BE = 256, UPB = 4;
};
template <>
struct Traits<V_Q6K> {
    static constexpr int BB = 210, BE = 256, UPB = 4;
};
template <>
struct Traits<V_Q80> {
    static constexpr int BB = 34, BE = 32, UPB = 1;
};
template <>
struct Traits<V_W8C> {
    static constexpr int BB = 32, BE = 32, UPB = 1;
};
template <>
struct Traits<V_W8A16> {
    static constexpr int BB = 34, BE = 32, UPB = 1;
};

// Shared-memory activation staging.
//   q8_1 variants: xs int8 codes | xd fp32 [M][K/32] | Q4_K: xm fp32 [M][K/32] = d*sum(q) (exact)
//                                                     | Q6_K: x16 int32 [M][K/16] = sum(q) per 16
//   W8A16       : xb bf16 [M][K/32 groups of 32, at a stride of 40 values]
// Staged activations are padded so that the 16-byte loads of the lanes of a row team fall in distinct
// shared-memory banks: K-quant codes in groups of 64 at a stride of 80 bytes, Q8_0 codes in groups of 32
// at 48 bytes, W8A16 bf16 values in groups of 32 at 80 bytes.  xrow is the padded bytes of one
// activation row.
template <int V>
struct XPad {
    static constexpr int GROUP = (V == V_Q4K || V == V_Q5K || V == V_Q6K) ? 64 : 32;  // codes (values) per group
    static constexpr int STRIDE = (V == V_Q80) ? 48 : 80;  // bytes
    __host__ __device__ static constexpr int row_bytes(int K) { return (K / GROUP) * STRIDE; }
    // byte offset of code e (e % 16 == 0 for 16-byte loads) within a padded row of codes
    __device__ static __forceinline__ int off(int e) { return (e / GROUP) * STRIDE + (e % GROUP); }
};

template <int V, int M>
struct XView {
    const int8_t* xs;
    const float* xd;
    const float* xm;
    const int* x16;
    const uint16_t* xb;
    int K;
    int xrow;  // padded bytes per activation row
    __device__ __forceinline__ XView(const uint8_t* base, int K_) : K(K_), xrow(XPad<V>::row_bytes(K_)) {
        if constexpr (V == V_W8A16 || V == V_W8C) {
            xb = reinterpret_cast<const uint16_t*>(base);
            xs = nullptr; xd = nullptr; xm = nullptr; x16 = nullptr;
        } else {
            xs = reinterpret_cast<const int8_t*>(base);
            xd = reinterpret_cast<const float*>(base + static_cast<size_t>(M) * xrow);
            xm = xd + M * (K >> 5);
            x16 = reinterpret_cast<const int*>(xm);
            xb = nullptr;
        }
    }
};

// Q6_K sums of 16 codes: for 32-value block idx (c = idx % 8 within its super-block, h = c / 4, k = c % 4)
// the terms of its halves t = 0, 1 are stored at 2 (idx - c) + 8h + 4t + k, so that a work unit
// (super-block, h, t) reads its four k values with one 16-byte load.  Each term is I2F_SEED - 32 * sum: the
// seed of the unit's dp4a chain, which takes the codes' +32 bias (sum (q-32) x = sum q x - 32 sum x) with it.
__device__ __forceinline__ int q6k_sum_pos(int idx, int t) {
    const int c = idx & 7;
    return 2 * (idx - c) + 8 * (c >> 2) + 4 * t + (c & 3);
}

// Store one staged q8_1 block (codes q[0..7], fp16 scale bits) for activation row i, block b.
template <int V, int M>
__device__ __forceinline__ void stage_codes(uint8_t* xsm, int K, int i, int b, const uint32_t (&q)[8]) {
    const int xrow = XPad<V>::row_bytes(K);
    uint4* dst = reinterpret_cast<uint4*>(xsm + i * xrow + XPad<V>::off(32 * b));
    dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
    dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
}

// Staging loads are issued XR rounds at a time before any of them is used, so the kernel pays one
// global-memory latency per XR rounds instead of one per round.  They are ordinary (L1-cached) loads:
// they run after the grid-dependency wait, which makes the producer's writes visible, and the 4-byte
// pieces of one q8_1 block then share one L1 line instead of going to L2 one by one.
constexpr int XR = 4;

template <int V, int M>
__device__ __forceinline__ void stage_one_q8_1(uint8_t* xsm, int K, int idx, uint32_t h, const uint32_t (&q)[8]) {
    const int nb = K >> 5;
    const int xrow = XPad<V>::row_bytes(K);
    float* xd = reinterpret_cast<float*>(xsm + static_cast<size_t>(M) * xrow);
    float* xm = xd + M * nb;
    int* x16 = reinterpret_cast<int*>(xm);
    const int i = idx / nb, b = idx - i * nb;
    stage_codes<V, M>(xsm, K, i, b, q);
    const float dx = h2f(h);
    xd[idx] = dx;
    if constexpr (V == V_Q4K || V == V_Q5K) {
        int sm = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) sm = dp4a(q[j], 0x01010101u, sm);
        xm[idx] = dx * static_cast<float>(sm);  // exact: 11-bit scale times |sum| <= 4064
    } else if constexpr (V == V_Q6K) {
        int s0 = 0, s1 = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) s0 = dp4a(q[j], 0x01010101u, s0);
#pragma unroll
        for (int j = 4; j < 8; ++j) s1 = dp4a(q[j], 0x01010101u, s1);
        x16[q6k_sum_pos(idx, 0)] = I2F_SEED - 32 * s0;
        x16[q6k_sum_pos(idx, 1)] = I2F_SEED - 32 * s1;
    }
}

// Activation rows a launch really has: M for the exact-m builds; the padded builds (the 16-row build for
// m = 9..16, and the K-chunk builds of 8 and 16 rows) stage rows m..M-1 as zeros and store none of their
// outputs.
template <int M, bool PADDED = false>
__device__ __forceinline__ int valid_rows(const GemvArgs& a) {
    if constexpr (M <= 8 && !PADDED) return M;
    else return a.m_rows;
}

// CHUNKED: the launch covers a K-chunk of each row ([x_col_off, x_col_off + K) of rows of x_row_stride
// values); otherwise the whole rows, x_row_stride == K.
template <int V, int M, bool CHUNKED>
__device__ __forceinline__ void stage_x(const GemvArgs& a, uint8_t* xsm, int tid, int nthreads) {
    const int K = a.K;
    if constexpr (V == V_W8A16 || V == V_W8C) {
        // bf16 kept as is: 8 values (one 16-byte load) per thread and round, into groups of 32 at 80 bytes
        const int xrow = XPad<V>::row_bytes(K);
        const uint4* src = reinterpret_cast<const uint4*>(a.x);
        const int n8 = (M * K) >> 3;
        const int n8_in = (valid_rows<M, CHUNKED>(a) * K) >> 3;  // rows past the call's m are staged as zeros
        for (int base = 0; base < n8; base += XR * nthreads) {
            uint4 v[XR];
#pragma unroll
            for (int r = 0; r < XR; ++r) {
                const int t = base + r * nthreads + tid;
                v[r] = make_uint4(0u, 0u, 0u, 0u);
                if (t < n8_in) {
                    if constexpr (!CHUNKED) v[r] = src[t];
                    else {
                        const int i = (8 * t) / K, e = 8 * t - i * K;
                        v[r] = src[(static_cast<size_t>(i) * a.x_row_stride + a.x_col_off + e) >> 3];
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < XR; ++r) {
                const int t = base + r * nthreads + tid;
                if (t < n8) {
                    const int i = (8 * t) / K, e = 8 * t - i * K;
                    *reinterpret_cast<uint4*>(xsm + i * xrow + (e >> 5) * 80 + 2 * (e & 31)) = v[r];
                }
            }
        }
    } else {
        const int nb = K >> 5;
        const int xrow = XPad<V>::row_bytes(K);
        float* xd = reinterpret_cast<float*>(xsm + static_cast<size_t>(M) * xrow);
        float* xm = xd + M * nb;
        int* x16 = reinterpret_cast<int*>(xm);
        const int nin = valid_rows<M, CHUNKED>(a) * nb;  // blocks of the call's rows; the rest are staged as zeros
        // block of the source rows that staged block idx (row i, block b of the chunk) comes from
        auto src_block = [&](int idx) -> size_t {
            if constexpr (!CHUNKED) return static_cast<size_t>(idx);
            const int i = idx / nb, b = idx - i * nb;
            return static_cast<size_t>(i) * (a.x_row_stride >> 5) + (a.x_col_off >> 5) + b;
        };
        if (a.act == ACT_Q8_1) {
            // One thread per staged q8_1 block (reads are L2 hits: the activation was just written).  The
            // single-row builds unroll two rounds (two blocks per thread cover rows of up to 16384 values),
            // a shorter staging code than four (measured: 4B-class sweep 1085 -> 1066 us).
            constexpr int XR = M == 1 ? 2 : qg::XR;
            for (int base = 0; base < M * nb; base += XR * nthreads) {
                uint32_t h[XR], q[XR][8];
#pragma unroll
                for (int r = 0; r < XR; ++r) {
                    const int idx = base + r * nthreads + tid;
                    h[r] = 0u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) q[r][j] = 0u;
                    if (idx < nin) {
                        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.x + src_block(idx) * 36);
                        h[r] = src[0];
#pragma unroll
                        for (int j = 0; j < 8; ++j) q[r][j] = src[1 + j];
                    }
                }
#pragma unroll
                for (int r = 0; r < XR; ++r) {
                    const int idx = base + r * nthreads + tid;
                    if (idx < M * nb) stage_one_q8_1<V, M>(xsm, K, idx, h[r], q[r]);
                }
            }
        } else {
            // fp32 activations, quantized here with the quantizer's arithmetic (8 lanes per block, four
            // values each, shuffle reductions inside the 8-lane group).  CTA 0 may also publish the blocks.
            const float4* xf = reinterpret_cast<const float4*>(a.x);
            const int part = tid & 7;
            uint8_t* out = blockIdx.x == 0 ? a.xq_out : nullptr;
            const int per_round = nthreads >> 3;
            // fp32 rounds move 16 bytes per lane: the single-row builds keep eight of them in flight; the
            // m-row builds, which fold the quantizer only into launches of at most a few thousand values,
            // take one at a time and stay smaller (measured: the 4B-class m = 8 sweep 2443 -> 2385 us)
            constexpr int XRF = M == 1 ? 2 * XR : 1;
            for (int base0 = 0; base0 < M * nb; base0 += XRF * per_round) {
                float4 vv[XRF];
#pragma unroll
                for (int r = 0; r < XRF; ++r) {
                    const int idx = base0 + r * per_round + (tid >> 3);
                    vv[r] = idx < nin ? xf[src_block(idx) * 8 + part] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int r = 0; r < XRF; ++r) {
                    if (base0 + r * per_round >= M * nb) break;  // uniform over the CTA: shuffles stay convergent
                    const int idx = base0 + r * per_round + (tid >> 3);
                    const bool valid = idx < M * nb;
                    const float4 v = vv[r];
                    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
                    const float d32 = __fdiv_rn(amax, 127.0f);
                    const int q0 = q8_1_code(v.x, d32), q1 = q8_1_code(v.y, d32);
                    const int q2 = q8_1_code(v.z, d32), q3 = q8_1_code(v.w, d32);
                    const uint32_t word = (static_cast<uint32_t>(q0) & 0xFFu) |
                                          ((static_cast<uint32_t>(q1) & 0xFFu) << 8) |
                                          ((static_cast<uint32_t>(q2) & 0xFFu) << 16) |
                                          ((static_cast<uint32_t>(q3) & 0xFFu) << 24);
                    const int sum4 = q0 + q1 + q2 + q3;
                    int half = sum4 + __shfl_xor_sync(0xffffffffu, sum4, 1);
                    half += __shfl_xor_sync(0xffffffffu, half, 2);  // sum over parts 0-3 or 4-7
                    const int sum = half + __shfl_xor_sync(0xffffffffu, half, 4);
                    if (valid) {
                        const int i = idx / nb, b = idx - i * nb;
                        *reinterpret_cast<uint32_t*>(xsm + i * xrow + XPad<V>::off(32 * b) + 4 * part) = word;
                        const __half dh = __float2half_rn(d32);
                        const float dx = __half2float(dh);
                        if (part == 0) {
                            xd[idx] = dx;
                            if constexpr (V == V_Q4K || V == V_Q5K) xm[idx] = dx * static_cast<float>(sum);
                            if constexpr (V == V_Q6K) x16[q6k_sum_pos(idx, 0)] = I2F_SEED - 32 * half;
                        }
                        if constexpr (V == V_Q6K) {
                            if (part == 4) x16[q6k_sum_pos(idx, 1)] = I2F_SEED - 32 * half;
                        }
                        if (out != nullptr && idx < nin) {
                            uint8_t* blk = out + src_block(idx) * 36;
                            reinterpret_cast<uint32_t*>(blk + 4)[part] = word;
                            if (part == 0) {
                                const __half sh = __float2half_rn(dx * static_cast<float>(sum));  // exact product
                                reinterpret_cast<uint32_t*>(blk)[0] =
                                    static_cast<uint32_t>(__half_as_ushort(dh)) |
                                    (static_cast<uint32_t>(__half_as_ushort(sh)) << 16);
                            }
                        }
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------------
// Per-format unit decoders.  `row` points at the first block of the staged copy in shared memory
// (2-byte aligned at least; 16-byte aligned for Q4_K and Q5_K), `u` is the unit index relative to it and `b0` the
// absolute index of that first block within the weight row.  acc[i] accumulates activation row i.

// One Q4_K unit of one weight row, decoded into registers: the codes of sub-blocks 2p (low nibbles) and
// 2p+1 (high nibbles, dotted in place: byte & 0xF0 = 16 * code, so their scale carries 1/16, exact), and
// the unit's scale and min factors.
struct Q4kUnit {
    uint32_t lo[8], hi[8];
    float dsc0, dsc1, dm0, dm1;
};

__device__ __forceinline__ Q4kUnit load_q4k(const uint8_t* blk, int p) {
    Q4kUnit w;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * p);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * p);
    const float d = h2f(hdr.x), dmin = h2f(hdr.x >> 16);
    const uint64_t s01 = static_cast<uint64_t>(hdr.y) | (static_cast<uint64_t>(hdr.z) << 32);
    const uint64_t s12 = static_cast<uint64_t>(hdr.z) | (static_cast<uint64_t>(hdr.w) << 32);
    const uint32_t sc12 = static_cast<uint32_t>(s01 >> (12 * p)) & 0xFFFu;        // sc[2p], sc[2p+1]
    const uint32_t mn12 = static_cast<uint32_t>(s12 >> (16 + 12 * p)) & 0xFFFu;   // mn[2p], mn[2p+1]
    w.dsc0 = d * i2f_small(static_cast<int>(sc12 & 63u));
    w.dsc1 = d * i2f_small(static_cast<int>(sc12 >> 6)) * 0.0625f;
    w.dm0 = dmin * i2f_small(static_cast<int>(mn12 & 63u));
    w.dm1 = dmin * i2f_small(static_cast<int>(mn12 >> 6));
    const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        w.lo[k] = q[k] & 0x0F0F0F0Fu;
        w.hi[k] = q[k] & 0xF0F0F0F0u;
    }
    return w;
}

// The unit's contribution to one activation row (its 64 staged codes x0..x3, block scales dx and the
// exact dx * sum(q) terms mx), added to v.
__device__ __forceinline__ float dot_q4k(const Q4kUnit& w, uint4 x0, uint4 x1, uint4 x2, uint4 x3, float2 dx,
                                         float2 mx, float v) {
    // four independent dp4a chains (lo/hi sub-block x two halves)
    int a0 = dp4a(w.lo[0], x0.x, 0), a1 = dp4a(w.lo[4], x1.x, 0);
    int c0 = dp4a_us(w.hi[0], x2.x, 0), c1 = dp4a_us(w.hi[4], x3.x, 0);
    a0 = dp4a(w.lo[1], x0.y, a0); a1 = dp4a(w.lo[5], x1.y, a1); c0 = dp4a_us(w.hi[1], x2.y, c0); c1 = dp4a_us(w.hi[5], x3.y, c1);
    a0 = dp4a(w.lo[2], x0.z, a0); a1 = dp4a(w.lo[6], x1.z, a1); c0 = dp4a_us(w.hi[2], x2.z, c0); c1 = dp4a_us(w.hi[6], x3.z, c1);
    a0 = dp4a(w.lo[3], x0.w, a0); a1 = dp4a(w.lo[7], x1.w, a1); c0 = dp4a_us(w.hi[3], x2.w, c0); c1 = dp4a_us(w.hi[7], x3.w, c1);
    v = fmaf(w.dsc0 * dx.x, i2f_small(a0 + a1), v);
    v = fmaf(w.dsc1 * dx.y, i2f_small(c0 + c1), v);
    v = fmaf(-w.dm0, mx.x, v);
    v = fmaf(-w.dm1, mx.y, v);
    return v;
}

// BR: u is already the block index (the single-row loop keeps it as an induction variable).
template <int M, bool BR = false>
__device__ __forceinline__ void unit_q4k(const uint8_t* row, int u, int lq, int b0, const XView<V_Q4K, M>& x,
                                         float (&acc)[M]) {
    const int br = BR ? u : u >> 2, p = lq;
    const int b = b0 + br;
    const Q4kUnit w = load_q4k(row + 144 * br, p);
    const int nb = x.K >> 5;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xw = reinterpret_cast<const uint4*>(x.xs + i * x.xrow + (4 * b + p) * 80);
        const int xb = i * nb + 8 * b + 2 * p;
        acc[i] = dot_q4k(w, xw[0], xw[1], xw[2], xw[3], *reinterpret_cast<const float2*>(x.xd + xb),
                         *reinterpret_cast<const float2*>(x.xm + xb), acc[i]);
    }
}

// The same unit of two weight rows against every activation row: each activation load serves both rows
// (the m-row kernels are bound by shared-memory load wavefronts), and each row's arithmetic is exactly
// that of unit_q4k.
template <int M>
__device__ __forceinline__ void unit_q4k_pair(const uint8_t* rowA, const uint8_t* rowB, int u, int lq, int b0,
                                              const XView<V_Q4K, M>& x, float (&accA)[M], float (&accB)[M]) {
    const int br = u >> 2, p = lq;
    const int b = b0 + br;
    const Q4kUnit wa = load_q4k(rowA + 144 * br, p);
    const Q4kUnit wb = load_q4k(rowB + 144 * br, p);
    const int nb = x.K >> 5;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xw = reinterpret_cast<const uint4*>(x.xs + i * x.xrow + (4 * b + p) * 80);
        const uint4 x0 = xw[0], x1 = xw[1], x2 = xw[2], x3 = xw[3];
        const int xb = i * nb + 8 * b + 2 * p;
        const float2 dx = *reinterpret_cast<const float2*>(x.xd + xb);
        const float2 mx = *reinterpret_cast<const float2*>(x.xm + xb);
        accA[i] = dot_q4k(wa, x0, x1, x2, x3, dx, mx, accA[i]);
        accB[i] = dot_q4k(wb, x0, x1, x2, x3, dx, mx, accB[i]);
    }
}

// Q5_K: as Q4_K (same header and qs packing at +48), with bit 4 of every code in qh[32] at +16: the unit
// of slice p (sub-blocks 2p, 2p+1) takes bits 2p and 2p+1 of each qh byte.
template <int M, bool BR = false>
__device__ __forceinline__ void unit_q5k(const uint8_t* row, int u, int lq, int b0, const XView<V_Q5K, M>& x,
                                         float (&acc)[M]) {
    const int br = BR ? u : u >> 2, p = lq;
    const uint8_t* blk = row + 176 * br;
    const int b = b0 + br;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4 h0 = *reinterpret_cast<const uint4*>(blk + 16);
    const uint4 h1 = *reinterpret_cast<const uint4*>(blk + 32);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 48 + 32 * p);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 64 + 32 * p);
    const float d = h2f(hdr.x), dmin = h2f(hdr.x >> 16);
    const uint64_t s01 = static_cast<uint64_t>(hdr.y) | (static_cast<uint64_t>(hdr.z) << 32);
    const uint64_t s12 = static_cast<uint64_t>(hdr.z) | (static_cast<uint64_t>(hdr.w) << 32);
    const uint32_t sc12 = static_cast<uint32_t>(s01 >> (12 * p)) & 0xFFFu;        // sc[2p], sc[2p+1]
    const uint32_t mn12 = static_cast<uint32_t>(s12 >> (16 + 12 * p)) & 0xFFFu;   // mn[2p], mn[2p+1]
    const float dsc0 = d * i2f_small(static_cast<int>(sc12 & 63u)), dsc1 = d * i2f_small(static_cast<int>(sc12 >> 6));
    const float dm0 = dmin * i2f_small(static_cast<int>(mn12 & 63u)), dm1 = dmin * i2f_small(static_cast<int>(mn12 >> 6));
    const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const uint32_t qh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t lo[8], hi[8];  // 5-bit codes of sub-blocks 2p and 2p+1
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t sh = qh[w] >> (2 * p);  // bit 0 of each byte: bit 2p; bit 1: bit 2p+1
        lo[w] = (q[w] & 0x0F0F0F0Fu) | ((sh << 4) & 0x10101010u);
        hi[w] = ((q[w] >> 4) & 0x0F0F0F0Fu) | ((sh << 3) & 0x10101010u);
    }
    const int nb = x.K >> 5;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xw = reinterpret_cast<const uint4*>(x.xs + i * x.xrow + (4 * b + p) * 80);
        const uint4 x0 = xw[0], x1 = xw[1], x2 = xw[2], x3 = xw[3];
        int a0 = dp4a(lo[0], x0.x, 0), a1 = dp4a(lo[4], x1.x, 0);
        int c0 = dp4a(hi[0], x2.x, 0), c1 = dp4a(hi[4], x3.x, 0);
        a0 = dp4a(lo[1], x0.y, a0); a1 = dp4a(lo[5], x1.y, a1); c0 = dp4a(hi[1], x2.y, c0); c1 = dp4a(hi[5], x3.y, c1);
        a0 = dp4a(lo[2], x0.z, a0); a1 = dp4a(lo[6], x1.z, a1); c0 = dp4a(hi[2], x2.z, c0); c1 = dp4a(hi[6], x3.z, c1);
        a0 = dp4a(lo[3], x0.w, a0); a1 = dp4a(lo[7], x1.w, a1); c0 = dp4a(hi[3], x2.w, c0); c1 = dp4a(hi[7], x3.w, c1);
        const int xb = i * nb + 8 * b + 2 * p;
        const float2 dx = *reinterpret_cast<const float2*>(x.xd + xb);
        const float2 mx = *reinterpret_cast<const float2*>(x.xm + xb);
        float v = acc[i];
        v = fmaf(dsc0 * dx.x, i2f_small(a0 + a1), v);
        v = fmaf(dsc1 * dx.y, i2f_small(c0 + c1), v);
        v = fmaf(-dm0, mx.x, v);
        v = fmaf(-dm1, mx.y, v);
        acc[i] = v;
    }
}

// One Q6_K unit of one weight row, decoded into registers: 16 codes (with the +32 bias) in each of the
// four sub-blocks 8h + 2k + tq, and their scales d * sc.
struct Q6kUnit {
    uint32_t q[4][4];
    float dsc[4];
};

// PH >= 0: the block's address mod 4 is known to be PH (a lane of the single-row loop keeps one phase for
// all its blocks), so the aligned base and the funnel shift are computed once instead of per load.
template <bool PH = false>
__device__ __forceinline__ Q6kUnit load_q6k(const uint8_t* blk, int h, int tq, uint32_t ph = 0) {
    Q6kUnit w;
    uint32_t la[4], lb[4], qh[4], scw[2];
    if constexpr (PH) {
        const uint32_t* a = reinterpret_cast<const uint32_t*>(blk - ph);
        const uint32_t sh = ph * 8u;
        lds_words_at<4>(a + 16 * h + 4 * tq, sh, la);
        lds_words_at<4>(a + 16 * h + 8 + 4 * tq, sh, lb);
        lds_words_at<4>(a + 32 + 8 * h + 4 * tq, sh, qh);
        lds_words_at<2>(a + 48 + 2 * h, sh, scw);
    } else {
        lds_words<4>(blk + 64 * h + 16 * tq, la);       // ql bytes 64h + t        (t = 16tq .. 16tq+15)
        lds_words<4>(blk + 64 * h + 32 + 16 * tq, lb);  // ql bytes 64h + 32 + t
        lds_words<4>(blk + 128 + 32 * h + 16 * tq, qh); // qh bytes 32h + t
        lds_words<2>(blk + 192 + 8 * h, scw);           // sc[8h .. 8h+7]
    }
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk + 208));
    // sub-scales of sub-blocks 8h + 2k + tq (k = 0..3): bytes tq and 2 + tq of each scale word
    const uint32_t sb0 = scw[0] ^ 0x80808080u, sb1 = scw[1] ^ 0x80808080u;
    w.dsc[0] = d * s8_to_f32(sb0, tq);
    w.dsc[1] = d * s8_to_f32(sb0, 2 + tq);
    w.dsc[2] = d * s8_to_f32(sb1, tq);
    w.dsc[3] = d * s8_to_f32(sb1, 2 + tq);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        w.q[0][k] = (la[k] & 0x0F0F0F0Fu) | ((qh[k] << 4) & 0x30303030u);
        w.q[1][k] = (lb[k] & 0x0F0F0F0Fu) | ((qh[k] << 2) & 0x30303030u);
        w.q[2][k] = ((la[k] >> 4) & 0x0F0F0F0Fu) | (qh[k] & 0x30303030u);
        w.q[3][k] = ((lb[k] >> 4) & 0x0F0F0F0Fu) | ((qh[k] >> 2) & 0x30303030u);
    }
    return w;
}

// The unit's contribution to one activation row: xv[k] holds the 16 staged codes of sub-block k, s16 the
// four chain seeds (I2F_SEED - 32 * code sum), dx4 the q8_1 scales.
__device__ __forceinline__ float dot_q6k(const Q6kUnit& w, const uint4 (&xv)[4], int4 s16, float4 dx4, float v) {
    const int sums[4] = {s16.x, s16.y, s16.z, s16.w};
    const float dxs[4] = {dx4.x, dx4.y, dx4.z, dx4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        int s = sums[k];
        s = dp4a(w.q[k][0], xv[k].x, s); s = dp4a(w.q[k][1], xv[k].y, s);
        s = dp4a(w.q[k][2], xv[k].z, s); s = dp4a(w.q[k][3], xv[k].w, s);
        v = fmaf(w.dsc[k] * dxs[k], seeded_to_f32(s), v);
    }
    return v;
}

// Staged activation operands of a Q6_K unit for activation row i.
template <int M>
__device__ __forceinline__ void q6k_act(const XView<V_Q6K, M>& x, int i, int b, int h, int tq, uint4 (&xv)[4],
                                        int4& s16, float4& dx4) {
    // codes 256b + 128h + 32k + 16tq: group 4b + 2h + k/2, offset 32(k&1) + 16tq
    const int8_t* xrow = x.xs + i * x.xrow + (4 * b + 2 * h) * 80 + 16 * tq;
#pragma unroll
    for (int k = 0; k < 4; ++k) xv[k] = *reinterpret_cast<const uint4*>(xrow + (k >> 1) * 80 + 32 * (k & 1));
    s16 = *reinterpret_cast<const int4*>(x.x16 + i * (x.K >> 4) + 16 * b + 8 * h + 4 * tq);
    dx4 = *reinterpret_cast<const float4*>(x.xd + i * (x.K >> 5) + 8 * b + 4 * h);
}

template <int M, bool BR = false>
__device__ __forceinline__ void unit_q6k(const uint8_t* row, int u, int lq, int b0, const XView<V_Q6K, M>& x,
                                         float (&acc)[M], uint32_t ph = 0) {
    const int br = BR ? u : u >> 2, h = lq >> 1, tq = lq & 1;
    const int b = b0 + br;
    const Q6kUnit w = load_q6k<BR>(row + 210 * br, h, tq, ph);
#pragma unroll
    for (int i = 0; i < M; ++i) {
        uint4 xv[4];
        int4 s16;
        float4 dx4;
        q6k_act<M>(x, i, b, h, tq, xv, s16, dx4);
        acc[i] = dot_q6k(w, xv, s16, dx4, acc[i]);
    }
}

// The same Q6_K unit of two weight rows against every activation row: each activation load serves both
// rows, and each row's arithmetic is exactly that of unit_q6k (rows stay bit-identical to calls without
// pairs).
template <int M>
__device__ __forceinline__ void unit_q6k_pair(const uint8_t* rowA, const uint8_t* rowB, int u, int lq, int b0,
                                              const XView<V_Q6K, M>& x, float (&accA)[M], float (&accB)[M]) {
    const int br = u >> 2, h = lq >> 1, tq = lq & 1;
    const int b = b0 + br;
    const Q6kUnit wa = load_q6k(rowA + 210 * br, h, tq);
    const Q6kUnit wb = load_q6k(rowB + 210 * br, h, tq);
#pragma unroll
    for (int i = 0; i < M; ++i) {
        uint4 xv[4];
        int4 s16;
        float4 dx4;
        q6k_act<M>(x, i, b, h, tq, xv, s16, dx4);
        accA[i] = dot_q6k(wa, xv, s16, dx4, accA[i]);
        accB[i] = dot_q6k(wb, xv, s16, dx4, accB[i]);
    }
}

// PH: the address phase (mod 4) of the block's codes is the lane's constant ph (single-row loop).
template <int M, bool PH = false>
__device__ __forceinline__ void unit_q80(const uint8_t* row, int br, int b0, const XView<V_Q80, M>& x, float (&acc)[M],
                                         uint32_t ph = 0) {
    const uint8_t* blk = row + 34 * br;
    const int b = b0 + br;
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk));
    uint32_t q[8];
    if constexpr (PH) lds_words_at<8>(reinterpret_cast<const uint32_t*>(blk + 2 - ph), ph * 8u, q);
    else lds_words<8>(blk + 2, q);
    const int nb = x.K >> 5;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xw = reinterpret_cast<const uint4*>(x.xs + i * x.xrow + 48 * b);
        const uint4 x0 = xw[0], x1 = xw[1];
        int s0 = dp4a(q[0], x0.x, I2F_SEED), s1 = dp4a(q[4], x1.x, 0);
        s0 = dp4a(q[1], x0.y, s0); s1 = dp4a(q[5], x1.y, s1);
        s0 = dp4a(q[2], x0.z, s0); s1 = dp4a(q[6], x1.z, s1);
        s0 = dp4a(q[3], x0.w, s0); s1 = dp4a(q[7], x1.w, s1);
        acc[i] = fmaf(d * x.xd[i * nb + b], seeded_to_f32(s0 + s1), acc[i]);
    }
}

// Two weights times two bf16 activations (one 32-bit word) accumulated into fp32.  A weight enters as
// the upper half of its exact fp32 value (an int8 has at most 8 significant bits, so that half is the
// exact bf16); the mixed-precision FMA rounds w * x + c once, like an fp32 FMA of the same values.
__device__ __forceinline__ void fma2_bf16(float w0, float w1, uint32_t x01, float& c0, float& c1) {
    asm("{\n\t.reg .b16 w0l, w0h, w1l, w1h, xl, xh;\n\t"
        "mov.b32 {w0l, w0h}, %2;\n\t"
        "mov.b32 {w1l, w1h}, %3;\n\t"
        "mov.b32 {xl, xh}, %4;\n\t"
        "fma.rn.f32.bf16 %0, w0h, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, w1h, xh, %1;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(w0), "f"(w1), "r"(x01));
}

// One Q8_0 block of one weight row as exact fp32 weights and the block scale.
struct W8Unit {
    float wf[32];
    float d;
};

template <bool PH = false>
__device__ __forceinline__ W8Unit load_w8a16(const uint8_t* blk, uint32_t ph = 0) {
    W8Unit w;
    w.d = h2f(*reinterpret_cast<const uint16_t*>(blk));
    uint32_t q[8];
    if constexpr (PH) lds_words_at<8>(reinterpret_cast<const uint32_t*>(blk + 2 - ph), ph * 8u, q);
    else lds_words<8>(blk + 2, q);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t v = q[k] ^ 0x80808080u;
#pragma unroll
        for (int j = 0; j < 4; ++j) w.wf[4 * k + j] = s8_to_f32(v, j);
    }
    return w;
}

// The block's contribution to one activation row (its 32 bf16 values in xx[0..3]).
__device__ __forceinline__ void dot8_w8a16(const W8Unit& w, int g, uint4 xx, float& p0, float& p1, float& p2,
                                           float& p3) {
    fma2_bf16(w.wf[8 * g + 0], w.wf[8 * g + 1], xx.x, p0, p1);
    fma2_bf16(w.wf[8 * g + 2], w.wf[8 * g + 3], xx.y, p2, p3);
    fma2_bf16(w.wf[8 * g + 4], w.wf[8 * g + 5], xx.z, p0, p1);
    fma2_bf16(w.wf[8 * g + 6], w.wf[8 * g + 7], xx.w, p2, p3);
}

__device__ __forceinline__ float dot_w8a16(const W8Unit& w, uint4 x0, uint4 x1, uint4 x2, uint4 x3, float acc) {
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;  // 8 values per 16-byte load
    dot8_w8a16(w, 0, x0, p0, p1, p2, p3);
    dot8_w8a16(w, 1, x1, p0, p1, p2, p3);
    dot8_w8a16(w, 2, x2, p0, p1, p2, p3);
    dot8_w8a16(w, 3, x3, p0, p1, p2, p3);
    return fmaf(w.d, (p0 + p1) + (p2 + p3), acc);
}

template <int M, bool PH = false>
__device__ __forceinline__ void unit_w8a16(const uint8_t* row, int br, int b0, const XView<V_W8A16, M>& x, float (&acc)[M],
                                           uint32_t ph = 0) {
    const W8Unit w = load_w8a16<PH>(row + 34 * br, ph);
    const int b = b0 + br;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xv = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(x.xb) + i * x.xrow + 80 * b);
        acc[i] = dot_w8a16(w, xv[0], xv[1], xv[2], xv[3], acc[i]);
    }
}

// Per-channel INT8 (one int8 per weight, no block scale; the row's fp32 scale is applied at the store):
// a unit is 32 consecutive weights (two aligned 16-byte loads), with the same exact int8 -> fp32 and
// mixed-precision FMA as unit_w8a16.
template <int M>
__device__ __forceinline__ void unit_w8c(const uint8_t* row, int br, int b0, const XView<V_W8C, M>& x, float (&acc)[M]) {
    const uint4 wa = *reinterpret_cast<const uint4*>(row + 32 * br);
    const uint4 wb = *reinterpret_cast<const uint4*>(row + 32 * br + 16);
    const int b = b0 + br;
    const uint32_t q[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    float wf[32];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t v = q[w] ^ 0x80808080u;
#pragma unroll
        for (int j = 0; j < 4; ++j) wf[4 * w + j] = s8_to_f32(v, j);
    }
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xv = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(x.xb) + i * x.xrow + 80 * b);
        float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint4 xx = xv[g];
            fma2_bf16(wf[8 * g + 0], wf[8 * g + 1], xx.x, p0, p1);
            fma2_bf16(wf[8 * g + 2], wf[8 * g + 3], xx.y, p2, p3);
            fma2_bf16(wf[8 * g + 4], wf[8 * g + 5], xx.z, p0, p1);
            fma2_bf16(wf[8 * g + 6], wf[8 * g + 7], xx.w, p2, p3);
        }
        acc[i] += (p0 + p1) + (p2 + p3);
    }
}

// BR: u is the unit's block index rather than its unit index (the same for the one-unit-per-block formats).
// ph (BR; Q6_K, Q8_0, W8A16): the address phase of the block (Q6_K) or of its codes (Q8_0, W8A16), mod 4, the
// same for every block of the lane.
template <int V, int M, bool BR = false>
__device__ __forceinline__ void decode_unit(const uint8_t* row, int u, int lq, int b0, const XView<V, M>& x,
                                            float (&acc)[M], uint32_t ph = 0) {
    if constexpr (V == V_Q4K) unit_q4k<M, BR>(row, u, lq, b0, x, acc);
    else if constexpr (V == V_Q5K) unit_q5k<M, BR>(row, u, lq, b0, x, acc);
    else if constexpr (V == V_Q6K) unit_q6k<M, BR>(row, u, lq, b0, x, acc, ph);
    else if constexpr (V == V_Q80) unit_q80<M, BR>(row, u, b0, x, acc, ph);
    else if constexpr (V == V_W8C) unit_w8c<M>(row, u, b0, x, acc);
    else unit_w8a16<M, BR>(row, u, b0, x, acc, ph);
}

// Two rows at once, for the formats and builds that pair rows (pair_rows).
template <int V, int M>
__device__ __forceinline__ void decode_pair(const uint8_t* rowA, const uint8_t* rowB, int u, int lq, const XView<V, M>& x,
                                            float (&accA)[M], float (&accB)[M]) {
    if constexpr (V == V_Q4K) unit_q4k_pair<M>(rowA, rowB, u, lq, 0, x, accA, accB);
    else if constexpr (V == V_Q6K) unit_q6k_pair<M>(rowA, rowB, u, lq, 0, x, accA, accB);
}

// ---------------------------------------------------------------------------------------------------

// ---------------------------------------------------------------------------------------------------
// Producer / consumer streaming.
//
// A CTA is NC consumer warps plus one producer warp.  The producer's lane 0 moves tiles of whole weight
// rows (16-48 KB) global -> shared with one bulk copy each (cp.async.bulk, L2 evict-first) into a ring of
// `stages` slots; slot s has a "full" mbarrier (completed by the copy's byte count) and an "empty"
// mbarrier (one arrival per consumer warp).  Consumers never meet at a CTA-wide barrier inside the loop:
// each warp waits for the slot to fill, decodes its rows, and signals the slot empty.  Rows are decoded
// by teams of L lanes (L <= 32, several rows per warp) or, for long rows, by G warps; a multi-warp team
// leaves one partial per warp in shared memory and the last warp to finish adds them in warp order, so
// the result does not depend on timing.  Tiles are dealt round-robin over the CTAs of a persistent grid.
// The producer issues its first tiles before the grid-dependency wait: under programmatic dependent launch
// the weight stream of this kernel overlaps the previous kernel, which never writes the weights.

// Argmax order, the one torch.argmax and numpy.argmax use: NaN above every number, then the larger value,
// and on equal values (or two NaNs) the smaller row.  The order is total, so the result is unique in any
// combining order.
__device__ __forceinline__ bool am_better(float v, int n, float bv, int bn) {
    const bool vn = v != v, bvn = bv != bv;
    if (vn || bvn) return vn && (!bvn || n < bn);
    return v > bv || (v == bv && n < bn);
}

// Output store: written, or (every K-chunk after the first) added to what the previous chunk wrote.
template <bool CHUNKED>
__device__ __forceinline__ void put_y(float* p, float v, int accumulate) {
    if constexpr (CHUNKED) {
        if (accumulate) v += *p;
    }
    *p = v;
}

// Matrix of the group that owns tile t.
__device__ __forceinline__ int group_of(const GemvArgs& a, int t) {
    int j = 0;
    while (j + 1 < a.count && t >= a.tile_start[j + 1]) ++j;
    return j;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// End of a fused-argmax launch: the CTA's best (value, row) per activation row goes to the scratch as one
// 8-byte pair; the last CTA to arrive combines all CTAs' pairs with all its consumer threads (at most a few
// independent loads each), writes the result and sets the arrival counter back to 0.  No thread waits for
// another CTA: the last arrival does the combine.
template <int M>
__device__ __forceinline__ void argmax_reduce_warps(float (&v)[M], int (&n)[M], float (*sv)[M], int (*sn)[M],
                                                    int warp, int lane_w) {
#pragma unroll
    for (int i = 0; i < M; ++i) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v[i], off);
            const int on = __shfl_xor_sync(0xffffffffu, n[i], off);
            if (am_better(ov, on, v[i], n[i])) { v[i] = ov; n[i] = on; }
        }
        if (lane_w == 0) {
            sv[warp][i] = v[i];
            sn[warp][i] = n[i];
        }
    }
}

template <int M>
__device__ __forceinline__ void argmax_finish(const GemvArgs& a, float (&bv)[M], int (&bn)[M], int warp, int lane_w,
                                           int NC) {
    __shared__ float sv[GEMV_CONSUMER_WARPS][M];
    __shared__ int sn[GEMV_CONSUMER_WARPS][M];
    __shared__ bool last;
    argmax_reduce_warps<M>(bv, bn, sv, sn, warp, lane_w);
    consumer_sync(NC * 32);
    unsigned* count = reinterpret_cast<unsigned*>(a.am_scratch);
    uint2* part = reinterpret_cast<uint2*>(a.am_scratch + AM_SCRATCH_HEAD);  // [gridDim.x][M] (value bits, row)
    if (warp == 0 && lane_w == 0) {
#pragma unroll
        for (int i = 0; i < M; ++i) {
            float v = sv[0][i];
            int n = sn[0][i];
            for (int w = 1; w < NC; ++w)
                if (am_better(sv[w][i], sn[w][i], v, n)) { v = sv[w][i]; n = sn[w][i]; }
            __stcg(part + blockIdx.x * M + i, make_uint2(__float_as_uint(v), static_cast<unsigned>(n)));
        }
        __threadfence();
        last = atomicAdd(count, 1u) == gridDim.x - 1;
    }
    consumer_sync(NC * 32);
    if (!last) return;
    __threadfence();
    const int t = warp * 32 + lane_w, nt = NC * 32, ncta = static_cast<int>(gridDim.x);
    constexpr int PER = 4;  // loads in flight per thread
#pragma unroll
    for (int i = 0; i < M; ++i) {
        bv[i] = -INFINITY;
        bn[i] = INT_MAX;
        for (int c0 = t; c0 < ncta; c0 += PER * nt) {
            uint2 p[PER];
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int c = c0 + j * nt;
                p[j] = c < ncta ? __ldcg(part + c * M + i) : make_uint2(__float_as_uint(-INFINITY), INT_MAX);
            }
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const float cv = __uint_as_float(p[j].x);
                const int cn = static_cast<int>(p[j].y);
                if (am_better(cv, cn, bv[i], bn[i])) { bv[i] = cv; bn[i] = cn; }
            }
        }
    }
    argmax_reduce_warps<M>(bv, bn, sv, sn, warp, lane_w);
    consumer_sync(NC * 32);
    if (warp == 0 && lane_w == 0) {
#pragma unroll
        for (int i = 0; i < M; ++i) {
            float v = sv[0][i];
            int n = sn[0][i];
            for (int w = 1; w < NC; ++w)
                if (am_better(sv[w][i], sn[w][i], v, n)) { v = sv[w][i]; n = sn[w][i]; }
            a.am_idx[i] = n == INT_MAX ? -1 : n;
            a.am_val[i] = v;
        }
        atomicExch(count, 0u);
    }
}

// Shared-memory ring of one CTA: `S` slots of `stage_bytes` with a "full" and an "empty" mbarrier each,
// and the arrival counters [MAX_STAGES][rstride] and partials [MAX_STAGES][rstride][G][M] of multi-warp
// row teams.
struct Ring {
    uint64_t* full;
    uint64_t* empty;
    uint8_t* slots;
    int* cnt;
    float* red;
    int S;
    unsigned stage_bytes;
    int rstride;
};

__device__ __forceinline__ Ring make_ring(uint8_t* smem, int S, unsigned stage_bytes, unsigned red_off, unsigned w_off,
                                          int rstride) {
    Ring r;
    r.full = reinterpret_cast<uint64_t*>(smem);
    r.empty = r.full + MAX_STAGES;
    r.slots = smem + w_off;
    r.cnt = reinterpret_cast<int*>(smem + red_off);
    r.red = reinterpret_cast<float*>(smem + red_off) + MAX_STAGES * rstride;
    r.S = S;
    r.stage_bytes = stage_bytes;
    r.rstride = rstride;
    return r;
}

// Barrier initialization and zeroed team counters; ends with a CTA-wide barrier.
__device__ __forceinline__ void ring_init(const Ring& r, int NC, int tid) {
    if (tid == 0) {
        for (int s = 0; s < r.S; ++s) {
            mbar_init(smem_addr(r.full + s), 1);
            mbar_init(smem_addr(r.empty + s), NC);
        }
        fence_mbar_init();
    }
    for (int t = tid; t < r.S * r.rstride; t += blockDim.x) r.cnt[t] = 0;
    __syncthreads();
}

// Producer lane: issues the tiles of launch `a` dealt to this CTA, continuing the ring position (k tiles
// issued so far, next slot s, the empty barriers' phases).  False after a wait that ran out (recorded).
template <bool CHUNKED>
__device__ __forceinline__ bool produce(const GemvArgs& a, const Ring& r, uint64_t pol, int& k, int& s,
                                        uint32_t& ephase) {
    for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++k) {
        if (k >= r.S) {
            const bool ok = mbar_wait_bounded(smem_addr(r.empty + s), (ephase >> s) & 1u);
            ephase ^= 1u << s;
            if (!ok) { atomicOr(a.err, ERR_WAIT_TIMEOUT); return false; }
        }
        const int j = group_of(a, t);
        const long long r0 = static_cast<long long>(t - a.tile_start[j]) * a.rows_per_tile;
        const int rows = static_cast<int>(min(static_cast<long long>(a.rows_per_tile), a.N[j] - r0));
        const uint8_t* W = a.W[j];
        uint8_t* slot = r.slots + s * r.stage_bytes;
        const long long lim = a.total_bytes[j] & ~15LL;
        if constexpr (!CHUNKED) {
            const long long s0 = r0 * a.row_bytes, e0 = s0 + rows * a.row_bytes;
            const long long al = s0 & ~15LL;
            const long long ce = min((e0 + 15) & ~15LL, lim);
            // Bytes past the last 16-byte boundary of the matrix cannot be bulk-copied (the copy would
            // read beyond the allocation): plain loads, before the arrival that publishes the slot.
            for (long long p = ce; p < e0; ++p) slot[p - al] = W[p];
            const uint32_t nbytes = static_cast<uint32_t>(ce - al);
            mbar_arrive_expect_tx(smem_addr(r.full + s), nbytes);
            if (nbytes) bulk_g2s(smem_addr(slot), W + al, nbytes, smem_addr(r.full + s), pol);
        } else {
            // K-chunked: one copy per row of the chunk's bytes (the aligned superset, as above), row rr at
            // rr * slot_row_stride in the slot; the arrival counts every copy's bytes.
            uint32_t nbytes = 0;
            for (int rr = 0; rr < rows; ++rr) {
                const long long s0 = (r0 + rr) * a.w_row_stride + a.w_col_off, e0 = s0 + a.row_bytes;
                const long long al = s0 & ~15LL, ce = min((e0 + 15) & ~15LL, lim);
                uint8_t* dst = slot + static_cast<size_t>(rr) * a.slot_row_stride;
                for (long long p = ce; p < e0; ++p) dst[p - al] = W[p];
                nbytes += static_cast<uint32_t>(ce - al);
            }
            mbar_arrive_expect_tx(smem_addr(r.full + s), nbytes);
            for (int rr = 0; rr < rows; ++rr) {
                const long long s0 = (r0 + rr) * a.w_row_stride + a.w_col_off, e0 = s0 + a.row_bytes;
                const long long al = s0 & ~15LL, ce = min((e0 + 15) & ~15LL, lim);
                if (ce > al)
                    bulk_g2s(smem_addr(slot + static_cast<size_t>(rr) * a.slot_row_stride), W + al,
                             static_cast<uint32_t>(ce - al), smem_addr(r.full + s), pol);
            }
        }
        if (++s == r.S) s = 0;
        // Only the first tiles go out before the grid dependency is met: a deeper prefetch competes for
        // HBM with the launches still on the critical path, the activation quantizer above all, whose
        // input read is a cold load (measured, 4B-class sweep: 1017 -> 983 us with one tile instead of
        // the whole ring).  A q8_1 activation comes from such a quantize launch; the other kinds come from
        // a GEMV or another producer, and there two tiles were better (W8A16 sweep 1114 -> 1105 us).
        if (k + 1 == (a.act == ACT_Q8_1 ? 1 : 2)) pdl_wait();
    }
    return true;
}

// Lets every copy this CTA issued land before the producer leaves (bounded).
__device__ __forceinline__ void producer_drain(const Ring& r, int issued, unsigned* err) {
    for (int j = (issued > r.S ? issued - r.S : 0); j < issued; ++j) {
        const int sj = j % r.S;
        if (!mbar_wait_bounded(smem_addr(r.full + sj), static_cast<uint32_t>((j / r.S) & 1)))
            atomicOr(err, ERR_DRAIN_TIMEOUT);
    }
}

// Consumer warps: decode the tiles of launch `a` dealt to this CTA against the activation staged at xsm,
// continuing the ring position (slot s, full-barrier phases).  ARGMAX keeps the running best row per
// activation row in bv / bn instead of writing y.  False after a wait that ran out (recorded).
template <int V, int M, bool ARGMAX, bool PAIR, bool CHUNKED>
__device__ __forceinline__ bool consume(const GemvArgs& a, const Ring& r, const uint8_t* xsm, int warp, int lane_w,
                                        int NC, int& s, uint32_t& fphase, float (&bv)[M], int (&bn)[M]) {
    const XView<V, M> xv(xsm, a.K);
    const int G = a.team_warps;
    int team, lane, L, T;
    if (G == 1) {
        L = 1 << a.lanes_log2;
        team = lane_w >> a.lanes_log2;  // team slot within the warp; rows are assigned per block below
        lane = lane_w & (L - 1);
        T = NC * (32 >> a.lanes_log2);
    } else {
        L = 32 * G;
        team = warp / G;
        lane = (warp % G) * 32 + lane_w;
        T = NC / G;
    }
    const int red_lanes = L < 32 ? L : 32;
    // A lane's units are lane, lane + L, ...: teams are a multiple of 4 lanes wide (the planner's rule), so
    // every unit of a lane has the same index mod 4, its part of a 256-value block in the K-quants, and the
    // offsets that follow from it stay out of the decode loop.
    const int lq = lane & 3;
    constexpr bool am = ARGMAX;  // fused argmax (the build for it) instead of writing y
    for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
        const bool ok = mbar_wait_bounded(smem_addr(r.full + s), (fphase >> s) & 1u);
        fphase ^= 1u << s;
#ifdef QGEMV_TRACE
        const int tix = (t - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x);
        unsigned long long* trc = a.trace && blockIdx.x < TRACE_CTAS && warp == 0 && lane_w == 0 && tix < 3
                                      ? a.trace + static_cast<size_t>(blockIdx.x) * TRACE_FIELDS : nullptr;
        if (trc) trc[8 + 2 * tix] = global_ns();
#endif
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane_w == 0) atomicOr(a.err, ERR_WAIT_TIMEOUT);
            return false;
        }
        const int j = group_of(a, t);
        const long long r0 = static_cast<long long>(t - a.tile_start[j]) * a.rows_per_tile;
        const int N = a.N[j];
        float* y = a.y[j];
        const int rows = static_cast<int>(min(static_cast<long long>(a.rows_per_tile), N - r0));
        const uint8_t* slot = r.slots + s * r.stage_bytes;
        const uint8_t* base = slot + ((r0 * a.row_bytes) & 15);
        // first byte of tile row rr in the slot (one contiguous copy, or one copy per row when K-chunked)
        auto row_at = [&](int rr) -> const uint8_t* {
            if constexpr (!CHUNKED) return base + rr * static_cast<int>(a.row_bytes);
            return slot + static_cast<size_t>(rr) * a.slot_row_stride + (((r0 + rr) * a.w_row_stride + a.w_col_off) & 15);
        };
        if (PAIR && a.row_pairs) {
            // Row pairs (lane-row teams, G == 1): a team decodes two consecutive rows unit by unit, so each
            // staged activation load serves both; every row's arithmetic (units, shuffle tree) is the
            // single-row path's, so rows are bit-identical to launches without pairs.
            for (int rb = 0; rb < rows; rb += 2 * T) {
                const int nblk = min(2 * T, rows - rb);
                const int npair = (nblk + 1) >> 1;
                const int ppw = (npair + NC - 1) / NC;
                const int pi = team < ppw ? warp * ppw + team : npair;
                const int rA = pi < npair ? rb + 2 * pi : rows;
                const int rB = rA + 1 < rb + nblk ? rA + 1 : rows;
                float accA[M], accB[M];
#pragma unroll
                for (int i = 0; i < M; ++i) accA[i] = accB[i] = 0.f;
                if (rA < rows) {
                    const uint8_t* rowA = row_at(rA);
                    const uint8_t* rowB = rB < rows ? row_at(rB) : rowA;
                    float accA2[M], accB2[M];
#pragma unroll
                    for (int i = 0; i < M; ++i) accA2[i] = accB2[i] = 0.f;
                    int u = lane;
#pragma unroll 1
                    for (; u + L < a.units_per_row; u += 2 * L) {
                        decode_pair<V, M>(rowA, rowB, u, lq, xv, accA, accB);
                        decode_pair<V, M>(rowA, rowB, u + L, lq, xv, accA2, accB2);
                    }
                    if (u < a.units_per_row) decode_pair<V, M>(rowA, rowB, u, lq, xv, accA, accB);
#pragma unroll
                    for (int i = 0; i < M; ++i) {
                        accA[i] += accA2[i];
                        accB[i] += accB2[i];
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    if (off < red_lanes) {
#pragma unroll
                        for (int i = 0; i < M; ++i) {
                            accA[i] += __shfl_xor_sync(0xffffffffu, accA[i], off);
                            accB[i] += __shfl_xor_sync(0xffffffffu, accB[i], off);
                        }
                    }
                }
                if (rA < rows && lane == 0) {
#pragma unroll
                    for (int i = 0; i < M; ++i) {
                        if ((M <= 8 && !CHUNKED) || i < a.m_rows) {
                            put_y<CHUNKED>(y + static_cast<size_t>(i) * N + r0 + rA, accA[i], a.accumulate);
                            if (rB < rows) put_y<CHUNKED>(y + static_cast<size_t>(i) * N + r0 + rB, accB[i], a.accumulate);
                        }
                    }
                }
            }
            __syncwarp();
#ifdef QGEMV_TRACE
            if (trc) trc[9 + 2 * tix] = global_ns();
#endif
            if (lane_w == 0) mbar_arrive(smem_addr(r.empty + s));
            if (++s == r.S) s = 0;
            continue;
        }
        for (int rb = 0; rb < rows; rb += T) {
            // Row of this team in the block [rb, rb + T): each warp takes a run of consecutive rows
            // (consecutive rows fall in different shared-memory banks); a partial block is spread over
            // all warps (shorter critical path for small matrices).
            int rr;
            if (G == 1) {
                const int nblk = min(T, rows - rb);
                const int rpw = (nblk + NC - 1) / NC;
                rr = team < rpw ? rb + warp * rpw + team : rows;
            } else {
                rr = rb + team;
            }
            float rs = 1.f;  // per-channel INT8: the output row's scale, loaded before the decode
            if constexpr (V == V_W8C) {
                if (rr < rows) rs = a.rscale[j][r0 + rr];
            }
            float acc[M];
#pragma unroll
            for (int i = 0; i < M; ++i) acc[i] = 0.f;
            if (rr < rows) {
                const uint8_t* row = row_at(rr);
                // Units lane, lane + L, ... in pairs with two accumulators (independent dependency chains),
                // summed at the end: the order depends on (units per row, L) only.
                float acc2[M];
#pragma unroll
                for (int i = 0; i < M; ++i) acc2[i] = 0.f;
                if constexpr (M == 1) {
                    // the block index as its own induction variable (unit u = lane + L j is in block
                    // lane / UPB + (L / UPB) j): shorter address arithmetic in the single-row builds
                    // Q6_K: with an even block step (teams of 8 lanes or more) every block of the lane has the
                    // address phase of its first block (210 bytes a block)
                    constexpr int UPB = Traits<V>::UPB;
                    const int bs = L / UPB;
                    int u = lane, br = lane / UPB;
                    // (Q8_0 and W8A16: the codes of 34-byte blocks, at a step of L blocks, L >= 4)
                    const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(
                                            V == V_Q6K ? row + 210 * br : row + 34 * br + 2)) & 3u;
                    if (V == V_Q6K && (bs & 1)) {
#pragma unroll 1
                        for (; u + L < a.units_per_row; u += 2 * L) {
                            decode_unit<V, M>(row, u, lq, 0, xv, acc);
                            decode_unit<V, M>(row, u + L, lq, 0, xv, acc2);
                        }
                        if (u < a.units_per_row) decode_unit<V, M>(row, u, lq, 0, xv, acc);
                    } else {
#pragma unroll 1
                        for (; u + L < a.units_per_row; u += 2 * L, br += 2 * bs) {
                            decode_unit<V, M, true>(row, br, lq, 0, xv, acc, ph);
                            decode_unit<V, M, true>(row, br + bs, lq, 0, xv, acc2, ph);
                        }
                        if (u < a.units_per_row) decode_unit<V, M, true>(row, br, lq, 0, xv, acc, ph);
                    }
                } else {
                    // the same order with the odd last unit folded into the loop (one copy of the m-row unit
                    // less: measured 4B-class m = 8 sweep 2383 -> 2361 us; the single-row builds are faster
                    // with the separate tail)
                    // (not the 8-row builds: measured 4B-class m = 8 sweep 2369 -> 2381 us with it, while m = 2,
                    // 4 and 16 gained 0.5-1.4%)
                    constexpr bool phased = (V == V_Q6K || V == V_Q80 || V == V_W8A16) && M != 8;
                    constexpr int UPB = Traits<V>::UPB;
                    const int bs = L / UPB;
                    if (phased && !(V == V_Q6K && (bs & 1))) {
                        // the formats of 2-byte-phase blocks: the lane's phase taken once, as in the single-row loop
                        int br = lane / UPB;
                        const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(
                                                V == V_Q6K ? row + 210 * br : row + 34 * br + 2)) & 3u;
#pragma unroll 1
                        for (int u = lane; u < a.units_per_row; u += 2 * L, br += 2 * bs) {
                            decode_unit<V, M, phased>(row, br, lq, 0, xv, acc, ph);
                            if (u + L < a.units_per_row) decode_unit<V, M, phased>(row, br + bs, lq, 0, xv, acc2, ph);
                        }
                    } else {
#pragma unroll 1
                        for (int u = lane; u < a.units_per_row; u += 2 * L) {
                            decode_unit<V, M>(row, u, lq, 0, xv, acc);
                            if (u + L < a.units_per_row) decode_unit<V, M>(row, u + L, lq, 0, xv, acc2);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < M; ++i) acc[i] += acc2[i];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                if (off < red_lanes) {
#pragma unroll
                    for (int i = 0; i < M; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
                }
            }
            if (rr < rows) {
                if (G == 1) {
                    if (lane == 0) {
                        const int n = static_cast<int>(r0) + rr;
#pragma unroll
                        for (int i = 0; i < M; ++i) {
                            const float v = acc[i] * rs;
                            if (!am) {
                                if ((M <= 8 && !CHUNKED) || i < a.m_rows) put_y<CHUNKED>(y + static_cast<size_t>(i) * N + n, v, a.accumulate);
                            } else if (am_better(v, n, bv[i], bn[i])) { bv[i] = v; bn[i] = n; }
                        }
                    }
                } else if (lane_w == 0) {
                    float* my = r.red + ((s * r.rstride + rr) * G + (warp % G)) * M;
#pragma unroll
                    for (int i = 0; i < M; ++i) my[i] = acc[i];
                    __threadfence_block();
                    const int prev = atomicAdd(r.cnt + s * r.rstride + rr, 1);
                    if (prev == G - 1) {
                        __threadfence_block();
                        const float* all = r.red + (s * r.rstride + rr) * G * M;
                        const int n = static_cast<int>(r0) + rr;
#pragma unroll
                        for (int i = 0; i < M; ++i) {
                            float v = 0.f;
                            for (int w = 0; w < G; ++w) v += all[w * M + i];
                            v *= rs;
                            if (!am) {
                                if ((M <= 8 && !CHUNKED) || i < a.m_rows) put_y<CHUNKED>(y + static_cast<size_t>(i) * N + n, v, a.accumulate);
                            } else if (am_better(v, n, bv[i], bn[i])) { bv[i] = v; bn[i] = n; }
                        }
                        r.cnt[s * r.rstride + rr] = 0;
                    }
                }
            }
        }
        __syncwarp();
#ifdef QGEMV_TRACE
        if (trc) trc[9 + 2 * tix] = global_ns();
#endif
        if (lane_w == 0) mbar_arrive(smem_addr(r.empty + s));
        if (++s == r.S) s = 0;
    }
    return true;
}

// PAIRS selects a build of its own with row pairs (the formats that pair rows only there: pair_build).
// CHUNKED selects the K-chunk builds (8 and 16 rows, padded like the 16-row build): each launch covers one
// chunk of every row (one copy per tile row, the activation chunk at a column offset) and adds to y after
// the first chunk.  They are separate instantiations so that the whole-row builds carry none of their code.
// STREAM selects the build for long single-row launches: no register cap (deeper software pipelining of
// the decode); the default single-row build is capped for four resident CTAs per SM.  Both builds run the
// same arithmetic in the same order.  ARGMAX (single-row streaming build only) reduces each activation
// row to its argmax instead of writing y.
template <int V, int M, bool STREAM = false, bool ARGMAX = false, bool CHUNKED = false, bool PAIRS = false>
__global__ void __launch_bounds__(GEMV_THREADS_MAX, (M == 1 && !STREAM) ? GEMV_MIN_CTAS_M1 : 0)
    gemv_staged_kernel(const GemvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
#ifdef QGEMV_TRACE
    const unsigned long long t_entry = global_ns();
    unsigned long long* tr =
        a.trace && blockIdx.x < TRACE_CTAS ? a.trace + static_cast<size_t>(blockIdx.x) * TRACE_FIELDS : nullptr;
#endif
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane_w = tid & 31;
    const int NC = (blockDim.x >> 5) - 1;
    const Ring r = make_ring(smem, a.stages, a.stage_bytes, a.red_off, a.w_off, a.rows_per_tile);
    ring_init(r, NC, tid);
    // The capped build (short single-row launches, up to four CTAs an SM) lets the next launch start only
    // once its activation is staged: an earlier start let a chain of short launches all prefetch at once
    // (measured, 0.6B-class sweep: 440.8 -> 433.8 us).  The other builds let it start at once.
    constexpr bool capped = M == 1 && !STREAM;
    if constexpr (!capped) pdl_launch_dependents();

    if (warp == NC) {
        // ---------------- producer ----------------
        if (lane_w == 0) {
            int k = 0, s = 0;
            uint32_t ephase = 0;
            const bool produced = produce<CHUNKED>(a, r, l2_evict_first_policy(), k, s, ephase);
#ifdef QGEMV_TRACE
            if (tr) tr[4] = global_ns();
#endif
            if (produced) producer_drain(r, k, a.err);
#ifdef QGEMV_TRACE
            if (tr) tr[5] = global_ns();
#endif
        }
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();
#ifdef QGEMV_TRACE
    if (tr && tid == 0) {
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        tr[0] = t_entry;
        tr[1] = global_ns();
        tr[6] = sm;
        tr[7] = 1;
    }
#endif
    stage_x<V, M, CHUNKED>(a, smem + a.x_off, tid, NC * 32);
    consumer_sync(NC * 32);
    if constexpr (capped) pdl_launch_dependents();
#ifdef QGEMV_TRACE
    if (tr && tid == 0) tr[2] = global_ns();
#endif
    float bv[M];
    int bn[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
        bv[i] = -INFINITY;
        bn[i] = INT_MAX;
    }
    int s = 0;
    uint32_t fphase = 0;
    // A wait that ran out ends the loop early; the argmax epilogue still runs (its barrier covers every
    // consumer warp, and the arrival counter must reach the grid size to reset itself).
    constexpr bool pairs = (pair_rows(V, M) || PAIRS) && !ARGMAX;
    consume<V, M, ARGMAX, pairs, CHUNKED>(a, r, smem + a.x_off, warp, lane_w, NC, s, fphase, bv, bn);
    if constexpr (ARGMAX) argmax_finish<M>(a, bv, bn, warp, lane_w, NC);
#ifdef QGEMV_TRACE
    consumer_sync(NC * 32);
    if (tr && tid == 0) tr[3] = global_ns();
#endif
}

}  // namespace qg
