// libqgemv C ABI: argument validation, per-device cache, launch planner, launches.
// Every check runs on the host before anything is enqueued; a non-zero status means nothing launched.
#include <atomic>
#include <mutex>
#include <unordered_map>
#include <stdint.h>
#include <string.h>

#include "../../include/qgemv.h"
#include "internal.h"

namespace qg {

const void* gemv_kernel_ptr_q4k(int kind);
const void* gemv_kernel_ptr_q6k(int kind);
const void* gemv_kernel_ptr_q80(int kind);
const void* gemv_kernel_ptr_w8a16(int kind);
const void* gemv_kernel_ptr_q5k(int kind);
const void* gemv_kernel_ptr_w8c(int kind);

const void* gemv_kernel_ptr(int variant, int kind) {
    switch (variant) {
    case V_Q4K: return gemv_kernel_ptr_q4k(kind);
    case V_Q6K: return gemv_kernel_ptr_q6k(kind);
    case V_Q80: return gemv_kernel_ptr_q80(kind);
    case V_W8A16: return gemv_kernel_ptr_w8a16(kind);
    case V_Q5K: return gemv_kernel_ptr_q5k(kind);
    case V_W8C: return gemv_kernel_ptr_w8c(kind);
    }
    return nullptr;
}

struct Geometry {
    int block_bytes, block_elems, units_per_block;
};

static Geometry geometry(int variant) {
    switch (variant) {
    case V_Q4K: return {144, 256, 4};
    case V_Q5K: return {176, 256, 4};
    case V_Q6K: return {210, 256, 4};
    case V_W8C: return {32, 32, 1};
    default: return {34, 32, 1};
    }
}

static unsigned round_up(unsigned v, unsigned a) { return (v + a - 1) / a * a; }

unsigned x_stage_bytes(int variant, int m, int K) {
    const size_t mk = static_cast<size_t>(m) * K;
    size_t b;
    const size_t padded = static_cast<size_t>(m) * (K / 64) * 80;  // codes in 80-byte groups of 64
    switch (variant) {
    case V_Q4K:
    case V_Q5K: b = padded + 4 * (mk / 32) * 2; break;            // codes, scales, scale*sum
    case V_Q6K: b = padded + 4 * (mk / 32) + 4 * (mk / 16); break;  // codes, scales, per-16 sums
    case V_Q80: b = static_cast<size_t>(m) * (K / 32) * 48 + 4 * (mk / 32); break;  // codes (48-byte groups), scales
    default: b = static_cast<size_t>(m) * (K / 32) * 80; break;                   // bf16 (80-byte groups)
    }
    return round_up(static_cast<unsigned>(b), 128);
}

// Dynamic shared memory of one CTA: the sm_103 opt-in maximum (232448 bytes) less 1 KB kept for the
// kernels' static shared memory (the fused-argmax epilogue).
constexpr unsigned SMEM_CAP = 232448 - 1024;
// Single-row launches of at least this many weight bytes use the streaming kernel build.
constexpr long long STREAM_MIN_BYTES = 4ll << 20;
constexpr unsigned BAR_BYTES = 2 * MAX_STAGES * 8;  // full + empty mbarrier per ring slot

static unsigned slot_bytes(long long tile_bytes) {
    return tile_bytes > (1LL << 30) ? (1u << 31) : round_up(static_cast<unsigned>(tile_bytes) + 48, 128);
}

// Slot bytes per row of a K-chunked tile: each row's chunk arrives as its own copy of the aligned superset
// (at most rb + 30 bytes), at a 16-byte aligned offset.
static long long seg_stride(long long rb) { return (rb + 32 + 15) / 16 * 16; }

// K limit of every entry point: rows longer than one pass of activation staging run as K-chunks.
constexpr int MAX_K_SERVED = 131072;

constexpr long long TILE_TARGET = 24576;  // bulk copies this large stream at full HBM rate
constexpr long long TILE_MAX = 49152;

static int pick_lanes_log2(int units);

// Row-team shape for rows of `rb` bytes and `units` work units: lanes per row from the unit count; fewer,
// wider teams while a tile holding one row per team would exceed TILE_MAX; then whole warps per row (G)
// for long rows.  It depends on (format, K) only, never on N: a row's summation order is then the same in
// every launch, so grouped and single calls give bit-identical rows.
static void team_shape(int units, long long rb, int l2_force, int* l2_out, int* G_out) {
    constexpr int NC = GEMV_CONSUMER_WARPS;
    // at least 4 lanes per team: the K-quant decoders take a lane's part of each block (unit index mod 4)
    // as fixed for all its units
    int l2 = l2_force >= 2 ? l2_force : pick_lanes_log2(units);
    while (l2 < 5 && static_cast<long long>(NC) * (32 >> l2) * rb > TILE_MAX) ++l2;
    int G = 1;
    if (l2 == 5)
        while (G < NC && static_cast<long long>(NC / G) * rb > TILE_MAX) G *= 2;
    *l2_out = l2;
    *G_out = G;
}

// Shared memory of the multi-warp reduction area: a counter and G x m partials per (ring slot, row).
// Activation rows a kernel build is compiled for: m itself up to 8, the padded 16-row build above.
static int kernel_m(int m) { return m <= 8 ? m : MAX_M; }
// Rows of the K-chunk build that serves m rows (8 or 16; rows past m padded).
static int chunk_m(int m) { return m <= 8 ? 8 : MAX_M; }
static int rows_of(int m, bool chunked) { return chunked ? chunk_m(m) : kernel_m(m); }

static unsigned red_bytes(int G, long long R, int m) {
    return G > 1 ? round_up(static_cast<unsigned>(MAX_STAGES * R * 4 + MAX_STAGES * R * G * m * 4), 128) : 0;
}

// Largest K (a block multiple) for which the smallest plan fits in shared memory: the activation staging,
// the reduction area and a two-slot ring of one row each (one row's chunk each, with per-row copies, when
// `chunked`).  Computed once per (variant, m, chunked).
static int max_k_compute(int variant, int m, bool chunked) {
    const Geometry g = geometry(variant);
    int lo = 0;
    for (int K = g.block_elems; K <= (1 << 22); K += g.block_elems) {
        const int nb = K / g.block_elems;
        const long long rb = static_cast<long long>(nb) * g.block_bytes;
        int l2, G;
        team_shape(nb * g.units_per_block, rb, -1, &l2, &G);
        const int km = rows_of(m, chunked);
        const unsigned long long need = BAR_BYTES + red_bytes(G, 1, km) + x_stage_bytes(variant, km, K) +
                                        2ull * slot_bytes(chunked ? seg_stride(rb) : rb);
        if (need > SMEM_CAP) break;
        lo = K;
    }
    return lo;
}

// Largest K of one launch over whole rows at m rows (one pass of activation staging), or with `chunked`
// of one K-chunk launch.
static int launch_max_k(int variant, int m, bool chunked = false) {
    static std::atomic<int> cache[2][NUM_VARIANTS][MAX_M + 1];  // 0 = not computed yet (every limit is positive)
    if (variant < 0 || variant >= NUM_VARIANTS || m < 1 || m > MAX_M) return 0;
    int v = cache[chunked][variant][m].load(std::memory_order_relaxed);
    if (v == 0) {
        v = max_k_compute(variant, m, chunked);
        cache[chunked][variant][m].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Largest K served at m rows (every m): rows beyond one pass of staging run as K-chunks.
static int max_k(int variant, int m) {
    if (variant < 0 || variant >= NUM_VARIANTS || m < 1 || m > MAX_M) return 0;
    return MAX_K_SERVED;
}

// Values per K-chunk of a call: K itself when the rows take one pass of activation staging (for m > 8
// possibly as two launches of 8 and m - 8 rows), else the width of the chunks (a multiple of 256, all equal
// but the last), as few as fit; 0 for an invalid argument.
static int chunk_k(int variant, int m, int K) {
    if (K < 1 || K > max_k(variant, m)) return 0;
    if (K <= launch_max_k(variant, m)) return K;
    if (m > 8 && K <= launch_max_k(variant, 8)) return K;
    // bf16 activations take 2 bytes a value in shared memory: chunks of half the widest that fits leave room
    // for a deeper weight ring (measured at m = 8: 7168 x 16384 W8A16 233 -> 137 us; the q8_1 formats run
    // best with the widest chunks)
    const int wide = launch_max_k(variant, m, true) / (variant == V_W8A16 || variant == V_W8C ? 2 : 1);
    const int kc0 = wide / 256 * 256;
    if (kc0 < 256) return 0;
    const int n = (K + kc0 - 1) / kc0;
    return ((K + n - 1) / n + 255) / 256 * 256;
}

// ---------------------------------------------------------------------------------------------------
// Per-device state

struct Plan {
    GemvArgs a;
    int kind;  // kernel build: m (1..8), or 0 for the single-row streaming build
    int grid;
    int threads;
    unsigned smem;
};

struct DeviceInfo {
    std::unordered_map<unsigned long long, Plan> plans;  // (variant, m, N, K) -> plan
    bool ready = false;
    bool supported = false;
    int sms = 0;
    unsigned* err = nullptr;  // device address of g_err on this device
    bool attr_set[NUM_VARIANTS][NUM_KINDS] = {};
};

static std::mutex g_mu;
static DeviceInfo g_dev[64];

__device__ unsigned g_err;

static thread_local int t_last_cuda = 0;
static std::atomic<unsigned long long> g_routes[QGEMV_NUM_ROUTES];
static std::atomic<int> g_fail_status{0};
static std::atomic<int> g_fail_count{0};

// Records e for qgemv_last_cuda_error and clears the runtime's last-error state (a non-sticky error such as
// an invalid launch configuration would otherwise be reported again by the next call's launch check, or by
// the caller's own).
static int cuda_fail(cudaError_t e) {
    t_last_cuda = static_cast<int>(e);
    (void)cudaGetLastError();
    return QGEMV_ERR_CUDA;
}

// Returns a status; on success *out points at the initialized entry of the current device.
static int device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return QGEMV_ERR_DEVICE;
    DeviceInfo& d = g_dev[dev];
    std::lock_guard<std::mutex> lk(g_mu);
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        int optin = 0;
        if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_fail(e);
        d.supported = (major == 10 && minor == 3) && optin >= static_cast<int>(SMEM_CAP);
        d.sms = sms;
        if (d.supported) {
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_err)) != cudaSuccess) return cuda_fail(e);
            d.err = static_cast<unsigned*>(p);
        }
        d.ready = true;
    }
    if (!d.supported) return QGEMV_ERR_DEVICE;
    *out = &d;
    return QGEMV_OK;
}

static bool take_injected_failure(int* status) {
    int c = g_fail_count.load();
    while (c > 0) {
        if (g_fail_count.compare_exchange_weak(c, c - 1)) {
            *status = g_fail_status.load();
            return true;
        }
    }
    return false;
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ---------------------------------------------------------------------------------------------------
// Planner: lanes per row, rows per tile, ring depth, grid.  A deterministic function of
// (variant, m, N, K, SM count).

static int pick_lanes_log2(int units) {
    // Short rows (<= 32 work units: K <= 2048 for the K-quants, K <= 1024 for Q8_0) come in matrices
    // small enough that a launch is latency-bound: about two units per lane keeps the serial decode
    // chain of a tile short.  Longer rows: every lane gets ~4 units per row (so per-row costs - the
    // shuffle reduction, the row loop - are spread over >= 128 weights), keeping >= 85% of the lanes
    // busy on the last pass.
    if (units <= 32) {
        int l2 = 2;
        while (l2 < 5 && (4 << l2) <= units) ++l2;
        return l2;
    }
    for (int l2 = 5; l2 >= 2; --l2) {
        const int L = 1 << l2;
        const int passes = (units + L - 1) / L;
        const double eff = static_cast<double>(units) / (L * passes);
        if (passes >= 4 && eff >= 0.85) return l2;
    }
    int best = 2;
    double best_eff = -1.0;
    for (int l2 = 2; l2 <= 5; ++l2) {
        const int L = 1 << l2;
        const double eff = static_cast<double>(units) / (L * ((units + L - 1) / L));
        if (eff > best_eff + 1e-9) { best_eff = eff; best = l2; }
    }
    return best;
}

// Tuning override (set through qgemv_tune_override; all zero = planner decides).
static std::atomic<int> g_ovr_l2{-1}, g_ovr_rows{0}, g_ovr_stages{0}, g_ovr_occ{0}, g_ovr_kind{0}, g_ovr_pairs{0};

// occ_override > 0 skips the occupancy query (host-only planning for introspection).
//
// Plan: row teams (lanes per row, or whole warps per row for long rows), tiles of R rows near
// TILE_TARGET bytes with every team holding a row, a ring deep enough to keep several tiles in flight
// while fitting two CTAs per SM when possible, and a persistent grid of at most SMs x resident CTAs.
// Small matrices get at least one tile per SM.
static int make_plan(int variant, int m, int N, int K, int sms, unsigned* err, int occ_override, Plan* p,
                     bool argmax = false, bool chunked = false) {
    const Geometry g = geometry(variant);
    const int nb = K / g.block_elems;
    const long long rb = static_cast<long long>(nb) * g.block_bytes;
    const long long trow = chunked ? seg_stride(rb) : rb;  // slot bytes per tile row
    const int units = nb * g.units_per_block;
    const int km = rows_of(m, chunked);                    // activation rows the kernel build stages
    const unsigned xb = x_stage_bytes(variant, km, K);
    constexpr int NC = GEMV_CONSUMER_WARPS;
    int l2, G;
    team_shape(units, rb, g_ovr_l2.load(), &l2, &G);
    const int force = g_ovr_kind.load();
    const bool stream = !argmax && !chunked && m == 1 && (force ? force == 2 : rb * N >= STREAM_MIN_BYTES);
    const long long teams = G == 1 ? static_cast<long long>(NC) * (32 >> l2) : NC / G;

    // Tile height, reduction area and ring depth; `pairs`: teams decode two rows at once, so a tile holds
    // two rows per team.
    struct Fit {
        long long R;
        unsigned red;
        int stages;
        unsigned long long smem;
        bool ok;
    };
    auto fit = [&](bool pairs) {
        Fit f;
        const long long tr = teams * (pairs ? 2 : 1);
        const long long kk = TILE_TARGET / (tr * trow);
        f.R = tr * (kk < 1 ? 1 : kk);
        // Small matrices: at least one tile per SM (latency regime; teams may idle).
        if ((N + f.R - 1) / f.R < sms) {
            const long long r2 = (N + sms - 1) / sms;
            if (r2 < f.R) f.R = r2 < 1 ? 1 : r2;
        }
        if (g_ovr_rows.load() > 0) f.R = g_ovr_rows.load();
        if (f.R > N) f.R = N;
        if (f.R < 1) f.R = 1;
        f.red = red_bytes(G, f.R, km);
        f.stages = g_ovr_stages.load() > 0 ? g_ovr_stages.load() : 4;
        if (f.stages > MAX_STAGES) f.stages = MAX_STAGES;
        auto need = [&](int st) {
            return BAR_BYTES + f.red + xb + static_cast<unsigned long long>(st) * slot_bytes(f.R * trow);
        };
        // Prefer two resident CTAs per SM, then accept one; long activations (large staging) take smaller
        // tiles before the plan gives up.
        while (f.stages > 2 && need(f.stages) > SMEM_CAP / 2) --f.stages;
        while (need(f.stages) > SMEM_CAP && f.R > 1) {
            f.R = (f.R + 1) / 2;
            f.red = red_bytes(G, f.R, km);
        }
        f.smem = need(f.stages);
        f.ok = f.smem <= SMEM_CAP;
        return f;
    };
    Fit f = fit(false);
    if (!f.ok) return QGEMV_ERR_UNSUPPORTED;
    // Single-row Q6_K launches of long rows (multi-warp teams): tiles of half the teams and a two-slot ring,
    // so that twice as many CTAs fit on an SM and a launch's tiles spread more evenly over the SMs.  Each
    // tile leaves half the teams of its CTA idle; the SM's other CTAs keep its decode busy.  Measured on one
    // box: the 2560 x 9728 down projection 8.70 -> 8.17 us, the 4B-class sweep 1061 -> 1044 us; W8A16 rows
    // (7168 x 16384, 16384 x 7168) ran slower this way (28.6 -> 32.6, 30.1 -> 31.7 us) and keep their plan.
    if (variant == V_Q6K && G > 1 && km == 1 && !chunked && g_ovr_rows.load() == 0 && g_ovr_stages.load() == 0 &&
        teams >= 2 && f.R == teams) {
        Fit h = f;
        h.R = teams / 2;
        h.red = red_bytes(G, h.R, km);
        h.stages = 2;
        h.smem = BAR_BYTES + h.red + xb + 2ull * slot_bytes(h.R * trow);
        h.ok = h.smem <= SMEM_CAP;
        if (h.ok) f = h;
    }
    bool pairs = false;
    const bool own_pair_build = pair_build(variant, km) && !chunked;
    if (!argmax && G == 1 && (pair_rows(variant, km) || own_pair_build)) {
        // Pairs pay when the tile still gives most teams a pair (measured: even where the larger tiles leave
        // one CTA per SM instead of two).
        const Fit fp = fit(true);
        const int mode = g_ovr_pairs.load();
        const bool good = fp.ok && (fp.R > teams || fp.R >= N);
        if (mode == 1 ? fp.ok : mode == 2 ? false : good) {
            f = fp;
            pairs = true;
        }
    }
    long long R = f.R;
    const unsigned red = f.red;
    const int stages = f.stages;
    auto need = [&](int st) {
        return BAR_BYTES + red + xb + static_cast<unsigned long long>(st) * slot_bytes(R * trow);
    };

    GemvArgs& a = p->a;
    a.row_bytes = rb;
    a.count = 1;
    a.N[0] = N;
    a.total_bytes[0] = rb * N;
    a.tile_start[0] = 0;
    a.tile_start[1] = static_cast<int>((N + R - 1) / R);
    a.K = K;
    a.rows_per_tile = static_cast<int>(R);
    a.num_tiles = static_cast<int>((N + R - 1) / R);
    a.units_per_row = units;
    a.lanes_log2 = l2;
    a.team_warps = G;
    a.stages = stages;
    a.stage_bytes = slot_bytes(R * trow);
    a.slot_row_stride = chunked ? static_cast<unsigned>(trow) : 0u;
    a.w_row_stride = rb;
    a.w_col_off = 0;
    a.x_row_stride = K;
    a.x_col_off = 0;
    a.accumulate = 0;
    a.red_off = BAR_BYTES;
    a.x_off = BAR_BYTES + red;
    a.w_off = BAR_BYTES + red + xb;
    a.err = err;
    p->smem = static_cast<unsigned>(need(stages));
    p->threads = GEMV_THREADS_MAX;
    // Single-row launches that stream many bytes use the build without the register cap: there the
    // decode rate, not the overlap of consecutive short launches, bounds the time.
    p->kind = m <= 8 ? m : KIND_M16;
    a.m_rows = m;
    a.row_pairs = pairs ? 1 : 0;
    if (argmax) p->kind = 9;  // the single-row streaming build with the fused argmax
    else if (chunked) p->kind = m <= 8 ? KIND_M8_CHUNK : KIND_M16_CHUNK;
    else if (stream) p->kind = 0;
    if (pairs && own_pair_build) p->kind = KIND_M8_PAIR;

    int occ = occ_override;
    if (occ < 1 && g_ovr_occ.load() > 0) occ = g_ovr_occ.load();
    if (occ < 1) {
        const void* fn = gemv_kernel_ptr(variant, p->kind);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, p->threads, p->smem) != cudaSuccess || occ < 1)
            occ = 1;
    }
    const long long cap = static_cast<long long>(sms) * occ;
    p->grid = static_cast<int>(a.num_tiles < cap ? a.num_tiles : cap);
    // the argmax scratch holds one partial per CTA; the grid is persistent, so fewer CTAs cover all tiles
    if (argmax && p->grid > static_cast<int>(AM_MAX_GRID)) p->grid = static_cast<int>(AM_MAX_GRID);
    return QGEMV_OK;
}

static int ensure_attr(DeviceInfo& dev, int variant, int kind) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev.attr_set[variant][kind]) return QGEMV_OK;
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel_ptr(variant, kind), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_CAP));
    if (e != cudaSuccess) return cuda_fail(e);
    dev.attr_set[variant][kind] = true;
    return QGEMV_OK;
}

cudaError_t launch_gemv(int variant, int kind, const GemvArgs& a, int grid, int threads, unsigned smem, bool pdl,
                        cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    GemvArgs copy = a;
    void* args[] = {&copy};
    cudaError_t e = cudaLaunchKernelExC(&cfg, gemv_kernel_ptr(variant, kind), args);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

// The part of each row one launch covers, for K-chunked calls: values [x_col_off, x_col_off + K) of rows of
// x_row_stride values and weight rows of w_row_stride bytes, the chunk at w_col_off bytes into each row;
// accumulate: add to y (every chunk after the first).
struct Chunk {
    long long w_row_stride, w_col_off;
    int x_row_stride, x_col_off, accumulate;
};

// One launch over `count` matrices that share the activation `x` (kind `act`); with `ch`, one K-chunk.
static int run_launch(int variant, int count, const void* const* W, float* const* y, const int* N, const void* x,
                      int act, void* xq_out, int m, int K, unsigned flags, void* stream, const float* const* rscale,
                      uint8_t* am_scratch, int* am_idx, float* am_val, const Chunk* ch) {
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st) return st;
    const bool argmax = am_scratch != nullptr;
    // shared-memory attribute of every build the planner may pick (the occupancy query needs it)
    if (ch) {
        if ((st = ensure_attr(*dev, variant, m <= 8 ? KIND_M8_CHUNK : KIND_M16_CHUNK))) return st;
    } else if ((st = ensure_attr(*dev, variant, m <= 8 ? m : KIND_M16))) return st;
    if (!ch && m == 1 && (st = ensure_attr(*dev, variant, 0))) return st;
    if (!ch && pair_build(variant, m) && (st = ensure_attr(*dev, variant, KIND_M8_PAIR))) return st;
    if (argmax && (st = ensure_attr(*dev, variant, 9))) return st;
    long long ntot = 0;
    for (int j = 0; j < count; ++j) ntot += N[j];
    if (ntot > (1LL << 30)) return QGEMV_ERR_UNSUPPORTED;
    const unsigned long long key = (static_cast<unsigned long long>(variant) << 59) |
                                   (static_cast<unsigned long long>(m) << 54) |
                                   (static_cast<unsigned long long>(ntot) << 24) | (argmax ? 1ull << 23 : 0ull) |
                                   (ch ? 1ull << 22 : 0ull) | static_cast<unsigned long long>(K);
    Plan p;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = dev->plans.find(key);
        if (it != dev->plans.end()) p = it->second;
        else {
            if ((st = make_plan(variant, m, static_cast<int>(ntot), K, dev->sms, dev->err, 0, &p, argmax,
                                ch != nullptr)))
                return st;
            dev->plans.emplace(key, p);
        }
    }
    GemvArgs& a = p.a;
    const long long R = a.rows_per_tile;
    a.count = count;
    if (ch) {
        a.w_row_stride = ch->w_row_stride;
        a.w_col_off = ch->w_col_off;
        a.x_row_stride = ch->x_row_stride;
        a.x_col_off = ch->x_col_off;
        a.accumulate = ch->accumulate;
    }
    int tiles = 0;
    for (int j = 0; j < count; ++j) {
        a.W[j] = static_cast<const uint8_t*>(W[j]);
        a.y[j] = y[j];
        a.rscale[j] = rscale ? rscale[j] : nullptr;
        a.N[j] = N[j];
        a.total_bytes[j] = a.w_row_stride * N[j];
        a.tile_start[j] = tiles;
        tiles += static_cast<int>((N[j] + R - 1) / R);
    }
    a.tile_start[count] = tiles;
    a.num_tiles = tiles;
    a.x = static_cast<const uint8_t*>(x);
    a.am_scratch = am_scratch;
    a.am_idx = am_idx;
    a.am_val = am_val;
    a.xq_out = static_cast<uint8_t*>(xq_out);
    a.act = act;
#ifdef QGEMV_TRACE
    a.trace = trace_next_launch();
#endif
    const int grid = p.grid < tiles ? p.grid : tiles;
    const bool pdl = (flags & QGEMV_FLAG_PDL) != 0;
    cudaError_t e = launch_gemv(variant, p.kind, a, grid, p.threads, p.smem, pdl, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    const int route0 = variant == V_Q5K ? QGEMV_ROUTE_Q5_K_M1 : variant == V_W8C ? QGEMV_ROUTE_W8A16_CHANNEL_M1 : 1 + variant * 8;
    g_routes[m <= 8 ? route0 + (m - 1) : QGEMV_ROUTE_M16].fetch_add(1, std::memory_order_relaxed);
    if (argmax) g_routes[QGEMV_ROUTE_ARGMAX].fetch_add(1, std::memory_order_relaxed);
    if (act == ACT_F32) g_routes[QGEMV_ROUTE_FUSED].fetch_add(1, std::memory_order_relaxed);
    if (count > 1) g_routes[QGEMV_ROUTE_GROUPED].fetch_add(1, std::memory_order_relaxed);
    if (pdl) g_routes[QGEMV_ROUTE_PDL].fetch_add(1, std::memory_order_relaxed);
    if (ch) g_routes[QGEMV_ROUTE_CHUNKED].fetch_add(1, std::memory_order_relaxed);
    return QGEMV_OK;
}

// A call over `count` matrices that share the activation `x` (kind `act`): one launch when the rows take one
// pass of activation staging; for m = 9..16 beyond the 16-row build's staging, launches of 8 and m - 8
// rows; beyond that, one launch per K-chunk (every launch after the first adds to y, in stream order).
static int run_gemv(int variant, int count, const void* const* W, float* const* y, const int* N, const void* x,
                    int act, void* xq_out, int m, int K, unsigned flags, void* stream,
                    const float* const* rscale = nullptr, uint8_t* am_scratch = nullptr, int* am_idx = nullptr,
                    float* am_val = nullptr) {
    const int kc = chunk_k(variant, m, K);
    if (kc == 0) return QGEMV_ERR_UNSUPPORTED;
    if (kc == K && m > 8 && K > launch_max_k(variant, m)) {
        // Beyond the 16-row build's activation staging: rows 0..7, then rows 8..m-1, as two launches.
        const size_t xrow = act == ACT_Q8_1 ? static_cast<size_t>(K / 32) * 36
                            : act == ACT_F32 ? static_cast<size_t>(K) * 4
                                             : static_cast<size_t>(K) * 2;
        float* y2[MAX_GROUP];
        for (int j = 0; j < count; ++j) y2[j] = y[j] + static_cast<size_t>(8) * N[j];
        int st = run_launch(variant, count, W, y, N, x, act, xq_out, 8, K, flags, stream, rscale, nullptr, nullptr,
                            nullptr, nullptr);
        if (st) return st;
        void* xq2 = xq_out ? static_cast<uint8_t*>(xq_out) + static_cast<size_t>(8) * (K / 32) * 36 : nullptr;
        return run_launch(variant, count, W, y2, N, static_cast<const uint8_t*>(x) + 8 * xrow, act, xq2, m - 8, K,
                          flags, stream, rscale, nullptr, nullptr, nullptr, nullptr);
    }
    if (kc == K)
        return run_launch(variant, count, W, y, N, x, act, xq_out, m, K, flags, stream, rscale, am_scratch, am_idx,
                          am_val, nullptr);
    if (am_scratch) return QGEMV_ERR_UNSUPPORTED;  // the fused argmax needs whole rows in one launch
    const Geometry g = geometry(variant);
    const long long full_rb = static_cast<long long>(K / g.block_elems) * g.block_bytes;
    for (int c0 = 0; c0 < K; c0 += kc) {
        const int kw = K - c0 < kc ? K - c0 : kc;
        const Chunk ch = {full_rb, static_cast<long long>(c0 / g.block_elems) * g.block_bytes, K, c0, c0 > 0};
        const int st = run_launch(variant, count, W, y, N, x, act, xq_out, m, kw, flags, stream, rscale, nullptr,
                                  nullptr, nullptr, &ch);
        if (st) return st;
    }
    return QGEMV_OK;
}

static int check_common(int m, int N, int K, int block_elems) {
    if (m < 1 || N < 1 || K < 1) return QGEMV_ERR_INVALID_ARG;
    if (K % block_elems) return QGEMV_ERR_INVALID_ARG;
    if (m > MAX_M) return QGEMV_ERR_UNSUPPORTED;
    return QGEMV_OK;
}

static int variant_of(int fmt) {
    switch (fmt) {
    case QGEMV_Q4_K: return V_Q4K;
    case QGEMV_Q6_K: return V_Q6K;
    case QGEMV_Q8_0: return V_Q80;
    case QGEMV_Q5_K: return V_Q5K;
    }
    return -1;
}

}  // namespace qg

using namespace qg;

extern "C" {

size_t qgemv_weight_bytes(int fmt, int N, int K) {
    const int v = variant_of(fmt);
    if (v < 0 || N < 1 || K < 1) return 0;
    const Geometry g = geometry(v);
    if (K % g.block_elems) return 0;
    return static_cast<size_t>(N) * static_cast<size_t>(K / g.block_elems) * g.block_bytes;
}

size_t qgemv_act_bytes(int m, int K) {
    if (m < 1 || K < 1 || K % 32) return 0;
    return static_cast<size_t>(m) * static_cast<size_t>(K / 32) * 36;
}

int qgemv_max_k(int fmt, int m) {
    const int v = variant_of(fmt);
    return v < 0 ? 0 : max_k(v, m);
}

int qgemv_max_k_w8a16(int m) { return max_k(V_W8A16, m); }

int qgemv_chunk_k(int fmt, int m, int K) {
    const int v = fmt == QGEMV_W8A16 ? V_W8A16 : fmt == QGEMV_W8A16_CHANNEL ? V_W8C : variant_of(fmt);
    if (v < 0 || m < 1 || m > MAX_M || K < 1 || K % geometry(v).block_elems) return 0;
    return chunk_k(v, m, K);
}

int qgemv_max_k_w8a16_channel(int m) { return max_k(V_W8C, m); }

const char* qgemv_status_string(int status) {
    switch (status) {
    case QGEMV_OK: return "QGEMV_OK";
    case QGEMV_ERR_INVALID_ARG: return "QGEMV_ERR_INVALID_ARG";
    case QGEMV_ERR_UNSUPPORTED: return "QGEMV_ERR_UNSUPPORTED";
    case QGEMV_ERR_MISALIGNED: return "QGEMV_ERR_MISALIGNED";
    case QGEMV_ERR_CUDA: return "QGEMV_ERR_CUDA";
    case QGEMV_ERR_DEVICE: return "QGEMV_ERR_DEVICE";
    case QGEMV_ERR_OVERLAP: return "QGEMV_ERR_OVERLAP";
    }
    return "QGEMV_ERR_UNKNOWN";
}

int qgemv_last_cuda_error(void) { return t_last_cuda; }

int qgemv_route_counts(unsigned long long* out, int n) {
    for (int i = 0; out && i < n && i < QGEMV_NUM_ROUTES; ++i) out[i] = g_routes[i].load();
    return QGEMV_NUM_ROUTES;
}

void qgemv_route_reset(void) {
    for (int i = 0; i < QGEMV_NUM_ROUTES; ++i) g_routes[i].store(0);
}

void qgemv_debug_fail_next(int status, int count) {
    g_fail_status.store(status);
    g_fail_count.store(count < 0 ? 0 : count);
}

int qgemv_device_error(unsigned int* out, int reset) {
    int st;
    if (take_injected_failure(&st)) return st;
    if (!out) return QGEMV_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev))) return st;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_err, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e);
    if (reset) {
        const unsigned zero = 0;
        if ((e = cudaMemcpyToSymbol(g_err, &zero, sizeof(unsigned))) != cudaSuccess) return cuda_fail(e);
    }
    return QGEMV_OK;
}

int qgemv_plan_info(int fmt, int m, int N, int K, int num_sms, int ctas_per_sm, long long* out) {
    const int v = fmt == QGEMV_W8A16 ? V_W8A16 : fmt == QGEMV_W8A16_CHANNEL ? V_W8C : variant_of(fmt);
    if (v < 0 || !out || num_sms < 1 || ctas_per_sm < 1) return QGEMV_ERR_INVALID_ARG;
    int st;
    if ((st = check_common(m, N, K, geometry(v).block_elems))) return st;
    const int kc = chunk_k(v, m, K);
    if (kc == 0) return QGEMV_ERR_UNSUPPORTED;
    const bool chunked = kc < K;
    if (!chunked && m > 8 && K > launch_max_k(v, m)) m = 8;  // served as launches of 8 and m - 8 rows: the first
    Plan p;                                                   // one's plan; K-chunked: the first chunk's plan
    if ((st = make_plan(v, m, N, kc, num_sms, nullptr, ctas_per_sm, &p, false, chunked))) return st;
    const long long vals[14] = {p.a.team_warps > 1 ? 32LL * p.a.team_warps : (1LL << p.a.lanes_log2),
                                p.a.rows_per_tile, p.a.num_tiles, p.a.stages, p.a.stage_bytes, p.smem, p.grid,
                                p.a.row_bytes, p.a.units_per_row, static_cast<long long>(p.a.w_off) - p.a.x_off,
                                p.threads, p.a.team_warps, static_cast<long long>(p.a.x_off) - p.a.red_off, p.kind};
    for (int i = 0; i < 14; ++i) out[i] = vals[i];
    return QGEMV_OK;
}

int qgemv_plan_info_chunk(int fmt, int m, int N, int Kc, int num_sms, int ctas_per_sm, long long* out) {
    const int v = fmt == QGEMV_W8A16 ? V_W8A16 : fmt == QGEMV_W8A16_CHANNEL ? V_W8C : variant_of(fmt);
    if (v < 0 || !out || num_sms < 1 || ctas_per_sm < 1) return QGEMV_ERR_INVALID_ARG;
    int st;
    if ((st = check_common(m, N, Kc, geometry(v).block_elems))) return st;
    if (Kc > launch_max_k(v, m, true)) return QGEMV_ERR_UNSUPPORTED;
    Plan p;
    if ((st = make_plan(v, m, N, Kc, num_sms, nullptr, ctas_per_sm, &p, false, true))) return st;
    const long long vals[15] = {p.a.team_warps > 1 ? 32LL * p.a.team_warps : (1LL << p.a.lanes_log2),
                                p.a.rows_per_tile, p.a.num_tiles, p.a.stages, p.a.stage_bytes, p.smem, p.grid,
                                p.a.row_bytes, p.a.units_per_row, static_cast<long long>(p.a.w_off) - p.a.x_off,
                                p.threads, p.a.team_warps, static_cast<long long>(p.a.x_off) - p.a.red_off, p.kind,
                                p.a.slot_row_stride};
    for (int i = 0; i < 15; ++i) out[i] = vals[i];
    return QGEMV_OK;
}

void qgemv_tune_pairs(int mode) { g_ovr_pairs.store(mode == 1 || mode == 2 ? mode : 0); }

void qgemv_tune_override(int ctas_per_sm, int lanes_log2, int rows_per_tile, int stages, int kernel_build) {
    g_ovr_occ.store(ctas_per_sm >= 1 && ctas_per_sm <= 4 ? ctas_per_sm : 0);
    g_ovr_kind.store(kernel_build == 1 || kernel_build == 2 ? kernel_build : 0);
    g_ovr_l2.store(lanes_log2 >= 0 && lanes_log2 <= 5 ? lanes_log2 : -1);
    g_ovr_rows.store(rows_per_tile > 0 ? rows_per_tile : 0);
    g_ovr_stages.store(stages >= 2 && stages <= MAX_STAGES ? stages : 0);
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& d : g_dev) d.plans.clear();
}

int qgemv_quantize_act_typed(int x_kind, const void* x, int m, int K, void* xq, unsigned flags, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    if (flags & ~(QGEMV_FLAG_PDL | QGEMV_FLAG_PDL_LATE_TRIGGER)) return QGEMV_ERR_INVALID_ARG;
    int xk;
    size_t esize;
    switch (x_kind) {
    case QGEMV_ACT_F32: xk = ACT_F32; esize = 4; break;
    case QGEMV_ACT_BF16: xk = ACT_BF16; esize = 2; break;
    case QGEMV_ACT_F16: xk = ACT_F16; esize = 2; break;
    default: return QGEMV_ERR_INVALID_ARG;
    }
    if ((st = check_common(m, 1, K, 32))) return st;
    if (!x || !xq) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(xq, 16)) return QGEMV_ERR_MISALIGNED;
    if (overlaps(x, static_cast<size_t>(m) * K * esize, xq, qgemv_act_bytes(m, K))) return QGEMV_ERR_OVERLAP;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev))) return st;
    const bool pdl = (flags & QGEMV_FLAG_PDL) != 0;
    const bool late = pdl && (flags & QGEMV_FLAG_PDL_LATE_TRIGGER) != 0;
    cudaError_t e =
        launch_quantize(xk, x, m, K, static_cast<uint8_t*>(xq), pdl, late, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    g_routes[0].fetch_add(1, std::memory_order_relaxed);
    if (pdl) g_routes[QGEMV_ROUTE_PDL].fetch_add(1, std::memory_order_relaxed);
    return QGEMV_OK;
}

int qgemv_quantize_act_ex(const float* x, int m, int K, void* xq, unsigned flags, void* stream) {
    return qgemv_quantize_act_typed(QGEMV_ACT_F32, x, m, K, xq, flags, stream);
}

int qgemv_quantize_act(const float* x, int m, int K, void* xq, void* stream) {
    return qgemv_quantize_act_ex(x, m, K, xq, 0u, stream);
}

static int multi_impl(int fmt, int count, const qgemv_mat* mats, int act_kind, const void* act, void* xq_out, int m,
                      int K, unsigned flags, void* stream);

int qgemv_multi(int fmt, int count, const qgemv_mat* mats, int act_kind, const void* act, void* xq_out, int m, int K,
                unsigned flags, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    return multi_impl(fmt, count, mats, act_kind, act, xq_out, m, K, flags, stream);
}

// Argument checks of a call over `count` matrices that share one activation; on success fills the
// variant and the per-matrix arrays.
static int validate_multi(int fmt, int count, const qgemv_mat* mats, int act_kind, const void* act, void* xq_out,
                          int m, int K, int* variant_out, const void** Ws, float** ys, int* Ns) {
    if (count < 1 || count > QGEMV_MAX_GROUP || !mats || !act) return QGEMV_ERR_INVALID_ARG;
    int variant;
    if (fmt == QGEMV_W8A16) {
        if (act_kind != QGEMV_ACT_BF16 || xq_out) return QGEMV_ERR_INVALID_ARG;
        variant = V_W8A16;
    } else {
        variant = variant_of(fmt);
        if (variant < 0 || (act_kind != QGEMV_ACT_Q8_1 && act_kind != QGEMV_ACT_F32)) return QGEMV_ERR_INVALID_ARG;
        if (xq_out && act_kind != QGEMV_ACT_F32) return QGEMV_ERR_INVALID_ARG;
    }
    const Geometry g = geometry(variant);
    if (m < 1 || K < 1 || K % g.block_elems) return QGEMV_ERR_INVALID_ARG;
    if (m > MAX_M) return QGEMV_ERR_UNSUPPORTED;
    const size_t act_bytes = act_kind == QGEMV_ACT_Q8_1 ? qgemv_act_bytes(m, K)
                             : act_kind == QGEMV_ACT_F32 ? static_cast<size_t>(m) * K * 4
                                                         : static_cast<size_t>(m) * K * 2;
    if (!aligned(act, 16) || (xq_out && !aligned(xq_out, 16))) return QGEMV_ERR_MISALIGNED;
    if (xq_out && overlaps(xq_out, qgemv_act_bytes(m, K), act, act_bytes)) return QGEMV_ERR_OVERLAP;
    for (int j = 0; j < count; ++j) {
        const qgemv_mat& q = mats[j];
        if (!q.W || !q.y || q.N < 1) return QGEMV_ERR_INVALID_ARG;
        if (!aligned(q.W, 16) || !aligned(q.y, 4)) return QGEMV_ERR_MISALIGNED;
        const size_t wb = static_cast<size_t>(q.N) * (K / g.block_elems) * g.block_bytes;
        const size_t yb = static_cast<size_t>(m) * q.N * 4;
        if (overlaps(q.y, yb, act, act_bytes)) return QGEMV_ERR_OVERLAP;
        if (xq_out && overlaps(q.y, yb, xq_out, qgemv_act_bytes(m, K))) return QGEMV_ERR_OVERLAP;
        for (int i = 0; i < count; ++i) {
            const size_t wi = static_cast<size_t>(mats[i].N) * (K / g.block_elems) * g.block_bytes;
            if (overlaps(q.y, yb, mats[i].W, wi)) return QGEMV_ERR_OVERLAP;
            if (i != j && overlaps(q.y, yb, mats[i].y, static_cast<size_t>(m) * mats[i].N * 4)) return QGEMV_ERR_OVERLAP;
        }
        if (xq_out && overlaps(xq_out, qgemv_act_bytes(m, K), q.W, wb)) return QGEMV_ERR_OVERLAP;
        Ws[j] = q.W;
        ys[j] = q.y;
        Ns[j] = q.N;
    }
    if (K > max_k(variant, m)) return QGEMV_ERR_UNSUPPORTED;
    *variant_out = variant;
    return QGEMV_OK;
}

static int multi_impl(int fmt, int count, const qgemv_mat* mats, int act_kind, const void* act, void* xq_out, int m,
                      int K, unsigned flags, void* stream) {
    if (flags & ~QGEMV_FLAG_PDL) return QGEMV_ERR_INVALID_ARG;
    const void* Ws[QGEMV_MAX_GROUP];
    float* ys[QGEMV_MAX_GROUP];
    int Ns[QGEMV_MAX_GROUP];
    int variant = 0;
    const int st = validate_multi(fmt, count, mats, act_kind, act, xq_out, m, K, &variant, Ws, ys, Ns);
    if (st) return st;
    const int ak = act_kind == QGEMV_ACT_Q8_1 ? ACT_Q8_1 : act_kind == QGEMV_ACT_F32 ? ACT_F32 : ACT_BF16;
    return run_gemv(variant, count, Ws, ys, Ns, act, ak, xq_out, m, K, flags, stream);
}

int qgemv_ex(int fmt, const void* W, const void* xq, float* y, int m, int N, int K, unsigned flags, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    const int v = variant_of(fmt);
    if (v < 0) return QGEMV_ERR_INVALID_ARG;
    if ((st = check_common(m, N, K, geometry(v).block_elems))) return st;
    if (!W || !xq || !y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(y, 4)) return QGEMV_ERR_MISALIGNED;
    if (K > max_k(v, m)) return QGEMV_ERR_UNSUPPORTED;
    const qgemv_mat mat = {W, y, N};
    if (overlaps(y, static_cast<size_t>(m) * N * 4, W, qgemv_weight_bytes(fmt, N, K)) ||
        overlaps(y, static_cast<size_t>(m) * N * 4, xq, qgemv_act_bytes(m, K)))
        return QGEMV_ERR_OVERLAP;
    return multi_impl(fmt, 1, &mat, QGEMV_ACT_Q8_1, xq, nullptr, m, K, flags, stream);
}

int qgemv(int fmt, const void* W, const void* xq, float* y, int m, int N, int K, void* stream) {
    return qgemv_ex(fmt, W, xq, y, m, N, K, 0u, stream);
}

int qgemv_w8a16_ex(const void* W, const void* x_bf16, float* y, int m, int N, int K, unsigned flags, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    if ((st = check_common(m, N, K, 32))) return st;
    if (!W || !x_bf16 || !y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(x_bf16, 16) || !aligned(y, 4)) return QGEMV_ERR_MISALIGNED;
    if (K > max_k(V_W8A16, m)) return QGEMV_ERR_UNSUPPORTED;
    const size_t wbytes = qgemv_weight_bytes(QGEMV_Q8_0, N, K);
    const size_t ybytes = static_cast<size_t>(m) * N * 4;
    if (overlaps(y, ybytes, W, wbytes) || overlaps(y, ybytes, x_bf16, static_cast<size_t>(m) * K * 2))
        return QGEMV_ERR_OVERLAP;
    const qgemv_mat mat = {W, y, N};
    return multi_impl(QGEMV_W8A16, 1, &mat, QGEMV_ACT_BF16, x_bf16, nullptr, m, K, flags, stream);
}

int qgemv_w8a16(const void* W, const void* x_bf16, float* y, int m, int N, int K, void* stream) {
    return qgemv_w8a16_ex(W, x_bf16, y, m, N, K, 0u, stream);
}

int qgemv_w8a16_channel_ex(const void* Wq, const float* scale, const void* x_bf16, float* y, int m, int N, int K,
                           unsigned flags, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    if (flags & ~QGEMV_FLAG_PDL) return QGEMV_ERR_INVALID_ARG;
    if ((st = check_common(m, N, K, 32))) return st;
    if (!Wq || !scale || !x_bf16 || !y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(Wq, 16) || !aligned(scale, 4) || !aligned(x_bf16, 16) || !aligned(y, 4)) return QGEMV_ERR_MISALIGNED;
    if (K > max_k(V_W8C, m)) return QGEMV_ERR_UNSUPPORTED;
    const size_t wbytes = static_cast<size_t>(N) * K, ybytes = static_cast<size_t>(m) * N * 4;
    if (overlaps(y, ybytes, Wq, wbytes) || overlaps(y, ybytes, x_bf16, static_cast<size_t>(m) * K * 2) ||
        overlaps(y, ybytes, scale, static_cast<size_t>(N) * 4))
        return QGEMV_ERR_OVERLAP;
    const void* Ws[1] = {Wq};
    float* ys[1] = {y};
    const int Ns[1] = {N};
    const float* ss[1] = {scale};
    return run_gemv(V_W8C, 1, Ws, ys, Ns, x_bf16, ACT_BF16, nullptr, m, K, flags, stream, ss);
}

size_t qgemv_argmax_scratch_bytes(int m) {
    if (m < 1 || m > 8) return 0;
    return AM_SCRATCH_HEAD + static_cast<size_t>(AM_MAX_GRID) * m * 8;
}

}  // extern "C"

// Checks of a fused-argmax call that need neither the scratch nor the device; on success *v_out is the
// kernel variant.
static int argmax_check(int fmt, const void* W, const void* xq, int m, int N, int K, const int* idx_out,
                        const float* val_out, unsigned flags, int* v_out) {
    if (flags & ~QGEMV_FLAG_PDL) return QGEMV_ERR_INVALID_ARG;
    const int v = variant_of(fmt);
    if (v < 0) return QGEMV_ERR_INVALID_ARG;
    int st;
    if ((st = check_common(m, N, K, geometry(v).block_elems))) return st;
    if (m != 1) return QGEMV_ERR_UNSUPPORTED;  // the fused argmax build is single-row
    if (!W || !xq || !idx_out || !val_out) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(idx_out, 4) || !aligned(val_out, 4))
        return QGEMV_ERR_MISALIGNED;
    if (K > launch_max_k(v, m)) return QGEMV_ERR_UNSUPPORTED;  // whole rows in one launch
    const size_t wbytes = qgemv_weight_bytes(fmt, N, K), xbytes = qgemv_act_bytes(m, K);
    const size_t ob = static_cast<size_t>(m) * 4;
    if (overlaps(idx_out, ob, W, wbytes) || overlaps(idx_out, ob, xq, xbytes) || overlaps(val_out, ob, W, wbytes) ||
        overlaps(val_out, ob, xq, xbytes) || overlaps(idx_out, ob, val_out, ob))
        return QGEMV_ERR_OVERLAP;
    *v_out = v;
    return QGEMV_OK;
}

extern "C" {

int qgemv_argmax(int fmt, const void* W, const void* xq, int m, int N, int K, void* scratch, size_t scratch_bytes,
                 int* idx_out, float* val_out, unsigned flags, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    int v = 0;
    if ((st = argmax_check(fmt, W, xq, m, N, K, idx_out, val_out, flags, &v))) return st;
    if (!scratch || scratch_bytes < qgemv_argmax_scratch_bytes(m)) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(scratch, 16)) return QGEMV_ERR_MISALIGNED;
    const size_t ob = static_cast<size_t>(m) * 4;
    if (overlaps(scratch, scratch_bytes, W, qgemv_weight_bytes(fmt, N, K)) ||
        overlaps(scratch, scratch_bytes, xq, qgemv_act_bytes(m, K)) || overlaps(scratch, scratch_bytes, idx_out, ob) ||
        overlaps(scratch, scratch_bytes, val_out, ob))
        return QGEMV_ERR_OVERLAP;
    const void* Ws[1] = {W};
    float* ys[1] = {nullptr};
    const int Ns[1] = {N};
    return run_gemv(v, 1, Ws, ys, Ns, xq, ACT_Q8_1, nullptr, m, K, flags, stream, nullptr,
                    static_cast<uint8_t*>(scratch), idx_out, val_out);
}

int qgemv_w8a16_channel(const void* Wq, const float* scale, const void* x_bf16, float* y, int m, int N, int K,
                        void* stream) {
    return qgemv_w8a16_channel_ex(Wq, scale, x_bf16, y, m, N, K, 0u, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------------
// qgemv_argmax on a library-owned scratch: a fixed array in static device memory (one instance per
// device, zero when the module loads), its address looked up once per device.

static __device__ __align__(256) uint8_t g_am_static[QGEMV_ARGMAX_STATIC_SCRATCH_BYTES];
static void* g_am_static_ptr[64];
static std::mutex g_am_static_mu;

extern "C" int qgemv_argmax_noalloc(int fmt, const void* W, const void* xq, int m, int N, int K, int* idx_out,
                                    float* val_out, unsigned flags, void* stream) {
    const size_t need = qgemv_argmax_scratch_bytes(m);
    if (need == 0) return QGEMV_ERR_INVALID_ARG;  // m outside 1..8
    if (need > QGEMV_ARGMAX_STATIC_SCRATCH_BYTES) return QGEMV_ERR_UNSUPPORTED;
    // Every host-side check, then the device check, before the symbol lookup touches the device: an
    // argument error returns its own status (not QGEMV_ERR_CUDA) and leaves no CUDA error behind.
    int v = 0, st;
    if ((st = argmax_check(fmt, W, xq, m, N, K, idx_out, val_out, flags, &v))) return st;
    DeviceInfo* info = nullptr;
    if ((st = device_info(&info))) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return QGEMV_ERR_DEVICE;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_am_static_mu);
        if (!g_am_static_ptr[dev]) {
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_am_static)) != cudaSuccess) return cuda_fail(e);
            g_am_static_ptr[dev] = p;
        }
        scratch = g_am_static_ptr[dev];
    }
    return qgemv_argmax(fmt, W, xq, m, N, K, scratch, QGEMV_ARGMAX_STATIC_SCRATCH_BYTES, idx_out, val_out, flags,
                        stream);
}

// ---------------------------------------------------------------------------------------------------
// Launch timeline (the traced build only; the normal build answers QGEMV_ERR_UNSUPPORTED).

#ifdef QGEMV_TRACE
namespace qg {
static __device__ unsigned long long g_trace[TRACE_LAUNCHES * TRACE_CTAS * TRACE_FIELDS];
static std::atomic<int> g_trace_seq{TRACE_LAUNCHES};  // numbering starts with qgemv_trace_begin

unsigned long long* trace_next_launch() {
    const int n = g_trace_seq.fetch_add(1);
    if (n < 0 || n >= TRACE_LAUNCHES) return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_trace) != cudaSuccess) return nullptr;
    return static_cast<unsigned long long*>(p) + static_cast<size_t>(n) * TRACE_CTAS * TRACE_FIELDS;
}
}  // namespace qg
#endif

extern "C" int qgemv_trace_info(int* launches, int* ctas, int* fields) {
#ifdef QGEMV_TRACE
    if (!launches || !ctas || !fields) return QGEMV_ERR_INVALID_ARG;
    *launches = TRACE_LAUNCHES;
    *ctas = TRACE_CTAS;
    *fields = TRACE_FIELDS;
    return QGEMV_OK;
#else
    (void)launches; (void)ctas; (void)fields;
    return QGEMV_ERR_UNSUPPORTED;
#endif
}

extern "C" int qgemv_trace_begin(void) {
#ifdef QGEMV_TRACE
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_trace);
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(g_trace));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    g_trace_seq.store(0);
    return QGEMV_OK;
#else
    return QGEMV_ERR_UNSUPPORTED;
#endif
}

extern "C" int qgemv_trace_read(unsigned long long* host, size_t bytes, int* launches) {
#ifdef QGEMV_TRACE
    if (!host || !launches || bytes > sizeof(g_trace)) return QGEMV_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyFromSymbol(host, g_trace, bytes);
    if (e != cudaSuccess) return cuda_fail(e);
    const int n = g_trace_seq.load();
    *launches = n < TRACE_LAUNCHES ? n : TRACE_LAUNCHES;
    return QGEMV_OK;
#else
    (void)host; (void)bytes; (void)launches;
    return QGEMV_ERR_UNSUPPORTED;
#endif
}
