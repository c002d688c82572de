// Staged decode-GEMV kernel for the block-quantized formats (sm_103a).
//
// Data path, per CTA (persistent; the grid covers the SMs):
//   1. The activation (q8_1 blocks, or bf16 for W8A16) is staged once into shared memory in a
//      decode-friendly form: codes contiguous per row, fp32 block scales, and per-format integer sums.
//   2. The weight stream is cut into warp work items (a few whole rows, or ~4 KB pieces of one long
//      row).  Each warp streams its own items global -> shared through a private ring of `stages` slots
//      with 16-byte cp.async copies (L2 evict-first), keeping stages-1 items in flight while it decodes
//      the current one.  Items that do not start on a 16-byte boundary (Q6_K / Q8_0 rows) are copied as
//      the aligned superset; the decoder indexes from the remainder.
//   3. Row teams of L lanes (L = 4..32) walk a row's work units; each unit dequantizes its codes in
//      registers, forms exact int32 dots with dp4a against the staged activation codes, and applies the
//      fp32 block scales.  Lane partials are reduced with xor-shuffles within the team.
//
// Work unit per format (64 weights for the K-quants, 32 for Q8_0):
//   Q4_K : one 32-byte slice g of qs -> sub-blocks 2g (low nibbles) and 2g+1 (high nibbles).
//   Q6_K : one half h of the block and 16 of its 32 qh columns -> 16 values in each of 4 sub-blocks.
//   Q8_0 : one block.
// This follows the "one warp per output row, dequantize in registers" decode of vllm.cpp PR #1936
// (the MMVQ geometry and T20 full-warp-cooperation sections), with the lanes-per-row made a plan
// parameter and the weight movement handed to the bulk-copy engine.
#pragma once
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
struct Traits<V_Q6K> {
    static constexpr int BB = 210, BE = 256, UPB = 4;
};
template <>
struct Traits<V_Q80> {
    static constexpr int BB = 34, BE = 32, UPB = 1;
};
template <>
struct Traits<V_W8A16> {
    static constexpr int BB = 34, BE = 32, UPB = 1;
};

// Shared-memory activation staging.
//   q8_1 variants: xs int8 [M][K] | xd fp32 [M][K/32] | Q4_K: xm fp32 [M][K/32] = d*sum(q) (exact)
//                                                     | Q6_K: x16 int32 [M][K/16] = sum(q) per 16
//   W8A16       : xf fp32 [M][K]
template <int V, int M>
struct XView {
    const int8_t* xs;
    const float* xd;
    const float* xm;
    const int* x16;
    const float* xf;
    int K;
    __device__ __forceinline__ XView(const uint8_t* base, int K_) : K(K_) {
        if constexpr (V == V_W8A16) {
            xf = reinterpret_cast<const float*>(base);
            xs = nullptr; xd = nullptr; xm = nullptr; x16 = nullptr;
        } else {
            xs = reinterpret_cast<const int8_t*>(base);
            xd = reinterpret_cast<const float*>(base + static_cast<size_t>(M) * K);
            xm = xd + M * (K >> 5);
            x16 = reinterpret_cast<const int*>(xm);
            xf = nullptr;
        }
    }
};

template <int V, int M>
__device__ __forceinline__ void stage_x(const GemvArgs& a, uint8_t* xsm) {
    const int K = a.K;
    if constexpr (V == V_W8A16) {
        float* xf = reinterpret_cast<float*>(xsm);
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.x);  // bf16 pairs
        const int n2 = (M * K) >> 1;
        for (int t = threadIdx.x; t < n2; t += blockDim.x) {
            const uint32_t v = __ldcg(src + t);
            xf[2 * t] = __uint_as_float(v << 16);
            xf[2 * t + 1] = __uint_as_float(v & 0xFFFF0000u);
        }
    } else {
        const int nb = K >> 5;
        int8_t* xs = reinterpret_cast<int8_t*>(xsm);
        float* xd = reinterpret_cast<float*>(xsm + static_cast<size_t>(M) * K);
        float* xm = xd + M * nb;
        int* x16 = reinterpret_cast<int*>(xm);
        for (int idx = threadIdx.x; idx < M * nb; idx += blockDim.x) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(a.x + static_cast<size_t>(idx) * 36);
            const uint32_t h = __ldcg(src);
            uint32_t q[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = __ldcg(src + 1 + j);
            const int i = idx / nb, b = idx - i * nb;
            uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(i) * K + 32 * b);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
            const float dx = h2f(h);
            xd[idx] = dx;
            if constexpr (V == V_Q4K) {
                int s = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) s = dp4a(q[j], 0x01010101u, s);
                xm[idx] = dx * static_cast<float>(s);  // exact: 11-bit scale times |s| <= 4064
            } else if constexpr (V == V_Q6K) {
                int s0 = 0, s1 = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) s0 = dp4a(q[j], 0x01010101u, s0);
#pragma unroll
                for (int j = 4; j < 8; ++j) s1 = dp4a(q[j], 0x01010101u, s1);
                x16[2 * idx] = s0;
                x16[2 * idx + 1] = s1;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------------
// Per-format unit decoders.  `row` points at the first block of the staged copy in shared memory
// (2-byte aligned at least; 16-byte aligned for Q4_K), `u` is the unit index relative to it and `b0` the
// absolute index of that first block within the weight row.  acc[i] accumulates activation row i.

template <int M>
__device__ __forceinline__ void unit_q4k(const uint8_t* row, int u, int b0, const XView<V_Q4K, M>& x, float (&acc)[M]) {
    const int br = u >> 2, p = u & 3;
    const uint8_t* blk = row + 144 * br;
    const int b = b0 + br;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * p);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * p);
    const float d = h2f(hdr.x), dmin = h2f(hdr.x >> 16);
    const uint64_t s01 = static_cast<uint64_t>(hdr.y) | (static_cast<uint64_t>(hdr.z) << 32);
    const uint64_t s12 = static_cast<uint64_t>(hdr.z) | (static_cast<uint64_t>(hdr.w) << 32);
    const uint32_t sc12 = static_cast<uint32_t>(s01 >> (12 * p)) & 0xFFFu;        // sc[2p], sc[2p+1]
    const uint32_t mn12 = static_cast<uint32_t>(s12 >> (16 + 12 * p)) & 0xFFFu;   // mn[2p], mn[2p+1]
    const float dsc0 = d * static_cast<float>(sc12 & 63u), dsc1 = d * static_cast<float>(sc12 >> 6);
    const float dm0 = dmin * static_cast<float>(mn12 & 63u), dm1 = dmin * static_cast<float>(mn12 >> 6);
    const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        lo[w] = q[w] & 0x0F0F0F0Fu;
        hi[w] = (q[w] >> 4) & 0x0F0F0F0Fu;
    }
    const int nb = x.K >> 5;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xw = reinterpret_cast<const uint4*>(x.xs + static_cast<size_t>(i) * x.K + 256 * b + 64 * p);
        const uint4 x0 = xw[0], x1 = xw[1], x2 = xw[2], x3 = xw[3];
        int s0 = 0, s1 = 0;
        s0 = dp4a(lo[0], x0.x, s0); s0 = dp4a(lo[1], x0.y, s0); s0 = dp4a(lo[2], x0.z, s0); s0 = dp4a(lo[3], x0.w, s0);
        s0 = dp4a(lo[4], x1.x, s0); s0 = dp4a(lo[5], x1.y, s0); s0 = dp4a(lo[6], x1.z, s0); s0 = dp4a(lo[7], x1.w, s0);
        s1 = dp4a(hi[0], x2.x, s1); s1 = dp4a(hi[1], x2.y, s1); s1 = dp4a(hi[2], x2.z, s1); s1 = dp4a(hi[3], x2.w, s1);
        s1 = dp4a(hi[4], x3.x, s1); s1 = dp4a(hi[5], x3.y, s1); s1 = dp4a(hi[6], x3.z, s1); s1 = dp4a(hi[7], x3.w, s1);
        const int xb = i * nb + 8 * b + 2 * p;
        const float2 dx = *reinterpret_cast<const float2*>(x.xd + xb);
        const float2 mx = *reinterpret_cast<const float2*>(x.xm + xb);
        float v = acc[i];
        v = fmaf(dsc0 * dx.x, static_cast<float>(s0), v);
        v = fmaf(dsc1 * dx.y, static_cast<float>(s1), v);
        v = fmaf(-dm0, mx.x, v);
        v = fmaf(-dm1, mx.y, v);
        acc[i] = v;
    }
}

template <int M>
__device__ __forceinline__ void unit_q6k(const uint8_t* row, int u, int b0, const XView<V_Q6K, M>& x, float (&acc)[M]) {
    const int br = u >> 2, h = (u >> 1) & 1, tq = u & 1;
    const uint8_t* blk = row + 210 * br;
    const int b = b0 + br;
    uint32_t la[4], lb[4], qh[4], scw[2];
    lds_words<4>(blk + 64 * h + 16 * tq, la);       // ql bytes 64h + t        (t = 16tq .. 16tq+15)
    lds_words<4>(blk + 64 * h + 32 + 16 * tq, lb);  // ql bytes 64h + 32 + t
    lds_words<4>(blk + 128 + 32 * h + 16 * tq, qh); // qh bytes 32h + t
    lds_words<2>(blk + 192 + 8 * h, scw);           // sc[8h .. 8h+7]
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk + 208));
    float dsc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int byte = 2 * k + tq;  // sub-block 8h + 2k + tq
        const uint32_t wsel = byte < 4 ? scw[0] : scw[1];
        const int sc = static_cast<int8_t>((wsel >> (8 * (byte & 3))) & 0xFFu);
        dsc[k] = d * static_cast<float>(sc);
    }
    uint32_t q[4][4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        q[0][w] = (la[w] & 0x0F0F0F0Fu) | ((qh[w] << 4) & 0x30303030u);
        q[1][w] = (lb[w] & 0x0F0F0F0Fu) | ((qh[w] << 2) & 0x30303030u);
        q[2][w] = ((la[w] >> 4) & 0x0F0F0F0Fu) | (qh[w] & 0x30303030u);
        q[3][w] = ((lb[w] >> 4) & 0x0F0F0F0Fu) | ((qh[w] >> 2) & 0x30303030u);
    }
    const int nb = x.K >> 5;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const int8_t* xrow = x.xs + static_cast<size_t>(i) * x.K + 256 * b + 128 * h + 16 * tq;
        const int* s16 = x.x16 + i * (x.K >> 4) + 16 * b + 8 * h + tq;
        const float* dxp = x.xd + i * nb + 8 * b + 4 * h;
        float v = acc[i];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xrow + 32 * k);
            int s = 0;
            s = dp4a(q[k][0], xv.x, s); s = dp4a(q[k][1], xv.y, s);
            s = dp4a(q[k][2], xv.z, s); s = dp4a(q[k][3], xv.w, s);
            s -= 32 * s16[2 * k];  // codes carry a +32 bias: sum (q-32) x = sum q x - 32 sum x
            v = fmaf(dsc[k] * dxp[k], static_cast<float>(s), v);
        }
        acc[i] = v;
    }
}

template <int M>
__device__ __forceinline__ void unit_q80(const uint8_t* row, int br, int b0, const XView<V_Q80, M>& x, float (&acc)[M]) {
    const uint8_t* blk = row + 34 * br;
    const int b = b0 + br;
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk));
    uint32_t q[8];
    lds_words<8>(blk + 2, q);
    const int nb = x.K >> 5;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const uint4* xw = reinterpret_cast<const uint4*>(x.xs + static_cast<size_t>(i) * x.K + 32 * b);
        const uint4 x0 = xw[0], x1 = xw[1];
        int s = 0;
        s = dp4a(q[0], x0.x, s); s = dp4a(q[1], x0.y, s); s = dp4a(q[2], x0.z, s); s = dp4a(q[3], x0.w, s);
        s = dp4a(q[4], x1.x, s); s = dp4a(q[5], x1.y, s); s = dp4a(q[6], x1.z, s); s = dp4a(q[7], x1.w, s);
        acc[i] = fmaf(d * x.xd[i * nb + b], static_cast<float>(s), acc[i]);
    }
}

// int8 byte j of v (v already xor 0x80808080, i.e. q + 128 unsigned) -> exact fp32 q:
// 0x4B0000uu is 2^23 + u as a float; subtracting 2^23 + 128 is exact.
__device__ __forceinline__ float s8_to_f32(uint32_t v_biased, int j) {
    return __uint_as_float(__byte_perm(v_biased, 0x4B000000u, 0x7650u | static_cast<unsigned>(j))) - 8388736.0f;
}

template <int M>
__device__ __forceinline__ void unit_w8a16(const uint8_t* row, int br, int b0, const XView<V_W8A16, M>& x, float (&acc)[M]) {
    const uint8_t* blk = row + 34 * br;
    const int b = b0 + br;
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk));
    uint32_t q[8];
    lds_words<8>(blk + 2, q);
    float wf[32];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t v = q[w] ^ 0x80808080u;
#pragma unroll
        for (int j = 0; j < 4; ++j) wf[4 * w + j] = s8_to_f32(v, j);
    }
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const float4* xv = reinterpret_cast<const float4*>(x.xf + static_cast<size_t>(i) * x.K + 32 * b);
        float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float4 xx = xv[w];
            p0 = fmaf(wf[4 * w + 0], xx.x, p0);
            p1 = fmaf(wf[4 * w + 1], xx.y, p1);
            p2 = fmaf(wf[4 * w + 2], xx.z, p2);
            p3 = fmaf(wf[4 * w + 3], xx.w, p3);
        }
        acc[i] = fmaf(d, (p0 + p1) + (p2 + p3), acc[i]);
    }
}

template <int V, int M>
__device__ __forceinline__ void decode_unit(const uint8_t* row, int u, int b0, const XView<V, M>& x, float (&acc)[M]) {
    if constexpr (V == V_Q4K) unit_q4k<M>(row, u, b0, x, acc);
    else if constexpr (V == V_Q6K) unit_q6k<M>(row, u, b0, x, acc);
    else if constexpr (V == V_Q80) unit_q80<M>(row, u, b0, x, acc);
    else unit_w8a16<M>(row, u, b0, x, acc);
}

// ---------------------------------------------------------------------------------------------------

// A position in a warp's sequence of copies: work item g (rows [g*R, g*R + R) or one row when rows are
// split), piece c of it, ring slot s.  Advanced incrementally (no division in the loop).
struct Cursor {
    int g, c, s;
    long long s0, e0;  // byte range [s0, e0) of the piece within the weight stream
};

template <int BB>
__device__ __forceinline__ void cursor_range(const GemvArgs& a, Cursor& q) {
    const long long rowstart = static_cast<long long>(q.g) * a.rows_per_tile * a.row_bytes;
    if (a.chunks == 1) {
        const int rows = min(a.rows_per_tile, a.N - q.g * a.rows_per_tile);
        q.s0 = rowstart;
        q.e0 = rowstart + static_cast<long long>(rows) * a.row_bytes;
    } else {
        const int c0 = q.c * a.chunk_blocks;
        const int c1 = min(a.blocks_per_row, c0 + a.chunk_blocks);
        q.s0 = rowstart + static_cast<long long>(c0) * BB;
        q.e0 = rowstart + static_cast<long long>(c1) * BB;
    }
}

template <int BB>
__device__ __forceinline__ void cursor_next(const GemvArgs& a, Cursor& q, int total_warps, int S) {
    if (++q.c == a.chunks) {
        q.c = 0;
        q.g += total_warps;
    }
    if (++q.s == S) q.s = 0;
    cursor_range<BB>(a, q);
}

// Whole warp: start moving bytes [s, e) of the weight stream into a ring slot as their 16-byte aligned
// superset, one 16-byte cp.async per lane and step (coalesced), then close this lane's copy group.
// Bytes past the last 16-byte boundary of the whole matrix cannot be copied in 16-byte pieces (that
// would read beyond the allocation); lane 0 moves them with plain loads (only the matrix's last copy).
__device__ __forceinline__ void warp_copy(const GemvArgs& a, long long s, long long e, uint8_t* slot, int lane,
                                          uint64_t pol) {
    const long long al = s & ~15LL;
    const long long ce = min((e + 15) & ~15LL, a.total_bytes & ~15LL);
    const int n16 = static_cast<int>((ce - al) >> 4);
    const uint32_t dst = smem_addr(slot);
    const uint8_t* src = a.W + al;
    for (int j = lane; j < n16; j += 32) cp_async16(dst + 16 * j, src + 16 * j, pol);
    if (lane == 0)
        for (long long p = ce; p < e; ++p) slot[p - al] = a.W[p];
    cp_async_commit();
}

// Warp-autonomous streaming.  Every warp owns a ring of `stages` slots in shared memory and keeps
// stages-1 copies of its own future work in flight with cp.async (the hardware tracks completion per
// lane: cp.async.wait_group, then a warp barrier so every lane sees every lane's bytes).  Work items
// (R rows, or one row cut into `chunks` pieces) are dealt round-robin over all warps of the grid.  The
// weight copies of the first stages-1 pieces are issued before the grid-dependency wait: with
// programmatic dependent launch they overlap the previous kernel, which never writes the weights.  The
// activation is staged after the wait; it is the only CTA-wide barrier.
template <int V, int M>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_staged_kernel(const GemvArgs a) {
    constexpr int BB = Traits<V>::BB, UPB = Traits<V>::UPB;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane_w = tid & 31;
    const int nwarps = blockDim.x >> 5;
    const int S = a.stages;
    const int C = a.chunks;
    uint8_t* ring = smem + a.w_off + static_cast<size_t>(warp) * S * a.stage_bytes;
    const int gwarp = blockIdx.x * nwarps + warp;
    const int total_warps = gridDim.x * nwarps;
    const uint64_t pol = l2_evict_first_policy();

    pdl_launch_dependents();
    // issue cursor: runs stages-1 pieces ahead of the decode cursor
    Cursor iq{gwarp, 0, 0, 0, 0};
    cursor_range<BB>(a, iq);
    for (int k = 0; k < S - 1; ++k) {
        if (iq.g < a.num_tiles) {
            warp_copy(a, iq.s0, iq.e0, ring + iq.s * a.stage_bytes, lane_w, pol);
            cursor_next<BB>(a, iq, total_warps, S);
        } else {
            cp_async_commit();
        }
    }
    pdl_wait();
    stage_x<V, M>(a, smem + a.x_off);
    __syncthreads();

    const XView<V, M> xv(smem + a.x_off, a.K);
    const int L = 1 << a.lanes_log2;
    const int team = lane_w >> a.lanes_log2;
    const int lane = lane_w & (L - 1);
    const int T = 32 >> a.lanes_log2;

    float acc[M];
#pragma unroll
    for (int i = 0; i < M; ++i) acc[i] = 0.f;
    Cursor q{gwarp, 0, 0, 0, 0};
    cursor_range<BB>(a, q);
    while (q.g < a.num_tiles) {
        if (iq.g < a.num_tiles) {
            warp_copy(a, iq.s0, iq.e0, ring + iq.s * a.stage_bytes, lane_w, pol);
            cursor_next<BB>(a, iq, total_warps, S);
        } else {
            cp_async_commit();
        }
        cp_async_wait_groups_except(S - 1);
        __syncwarp();

        const uint8_t* base = ring + q.s * a.stage_bytes + (q.s0 & 15);
        const int r0 = q.g * a.rows_per_tile;
        if (C == 1) {
            const int rows = min(a.rows_per_tile, a.N - r0);
            for (int rb = 0; rb < rows; rb += T) {
                const int rr = rb + team;
#pragma unroll
                for (int i = 0; i < M; ++i) acc[i] = 0.f;
                if (rr < rows) {
                    const uint8_t* row = base + rr * static_cast<int>(a.row_bytes);
#pragma unroll 2
                    for (int u = lane; u < a.units_per_row; u += L) decode_unit<V, M>(row, u, 0, xv, acc);
                }
                for (int off = L >> 1; off > 0; off >>= 1) {
#pragma unroll
                    for (int i = 0; i < M; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
                }
                if (rr < rows && lane == 0) {
#pragma unroll
                    for (int i = 0; i < M; ++i) a.y[static_cast<size_t>(i) * a.N + r0 + rr] = acc[i];
                }
            }
        } else {
            // One row per work item (whole warp, L = 32), streamed in `C` pieces; units are counted from
            // the first block of the piece.
            if (q.c == 0) {
#pragma unroll
                for (int i = 0; i < M; ++i) acc[i] = 0.f;
            }
            const int b0 = q.c * a.chunk_blocks;
            const int units = min(a.chunk_blocks, a.blocks_per_row - b0) * UPB;
#pragma unroll 2
            for (int u = lane_w; u < units; u += 32) decode_unit<V, M>(base, u, b0, xv, acc);
            if (q.c == C - 1) {
                float r[M];
#pragma unroll
                for (int i = 0; i < M; ++i) r[i] = acc[i];
                for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                    for (int i = 0; i < M; ++i) r[i] += __shfl_xor_sync(0xffffffffu, r[i], off);
                }
                if (lane_w == 0) {
#pragma unroll
                    for (int i = 0; i < M; ++i) a.y[static_cast<size_t>(i) * a.N + r0] = r[i];
                }
            }
        }
        __syncwarp();  // every lane is done with this slot before a later copy refills it
        cursor_next<BB>(a, q, total_warps, S);
    }
    cp_async_wait_all();
}

}  // namespace qg
