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

const void* gemv_kernel_ptr_q4k(int m);
const void* gemv_kernel_ptr_q6k(int m);
const void* gemv_kernel_ptr_q80(int m);
const void* gemv_kernel_ptr_w8a16(int m);

const void* gemv_kernel_ptr(int variant, int m) {
    switch (variant) {
    case V_Q4K: return gemv_kernel_ptr_q4k(m);
    case V_Q6K: return gemv_kernel_ptr_q6k(m);
    case V_Q80: return gemv_kernel_ptr_q80(m);
    case V_W8A16: return gemv_kernel_ptr_w8a16(m);
    }
    return nullptr;
}

struct Geometry {
    int block_bytes, block_elems, units_per_block;
};

static Geometry geometry(int variant) {
    switch (variant) {
    case V_Q4K: return {144, 256, 4};
    case V_Q6K: return {210, 256, 4};
    default: return {34, 32, 1};
    }
}

static unsigned round_up(unsigned v, unsigned a) { return (v + a - 1) / a * a; }

unsigned x_stage_bytes(int variant, int m, int K) {
    const size_t mk = static_cast<size_t>(m) * K;
    size_t b;
    switch (variant) {
    case V_Q4K: b = mk + 4 * (mk / 32) * 2; break;       // codes, scales, scale*sum
    case V_Q6K: b = mk + 4 * (mk / 32) + 4 * (mk / 16); break;  // codes, scales, per-16 sums
    case V_Q80: b = mk + 4 * (mk / 32); break;               // codes, scales
    default: b = 4 * mk; break;                              // fp32 activations
    }
    return round_up(static_cast<unsigned>(b), 128);
}

// Shared memory available to one CTA on sm_103 (opt-in maximum).
constexpr unsigned SMEM_CAP = 232448;
constexpr unsigned BAR_BYTES = (GEMV_THREADS / 32) * MAX_STAGES * 8;  // one mbarrier per ring slot per warp

static unsigned slot_bytes(long long tile_bytes) {
    return tile_bytes > (1LL << 30) ? (1u << 31) : round_up(static_cast<unsigned>(tile_bytes) + 48, 128);
}

// Largest K (a block multiple) whose activation staging plus two ring slots per warp fits in shared
// memory (long rows are streamed in chunks, so the slots do not grow with K beyond one chunk).
static int max_k(int variant, int m) {
    if (m < 1 || m > 8) return 0;
    const Geometry g = geometry(variant);
    const long long chunk = 2048 + g.block_bytes * (32 / g.units_per_block);
    int lo = 0;
    for (int K = g.block_elems; K <= (1 << 22); K += g.block_elems) {
        const long long rb = static_cast<long long>(K / g.block_elems) * g.block_bytes;
        const long long item = rb < chunk ? rb : chunk;
        const unsigned long long need = BAR_BYTES + x_stage_bytes(variant, m, K) +
                                        static_cast<unsigned long long>(GEMV_THREADS / 32) * 2 * slot_bytes(item);
        if (need > SMEM_CAP) break;
        lo = K;
    }
    return lo;
}

// ---------------------------------------------------------------------------------------------------
// Per-device state

struct Plan {
    GemvArgs a;
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
    bool attr_set[4][9] = {};
};

static std::mutex g_mu;
static DeviceInfo g_dev[64];

__device__ unsigned g_err;

static thread_local int t_last_cuda = 0;
static std::atomic<unsigned long long> g_routes[QGEMV_NUM_ROUTES];
static std::atomic<int> g_fail_status{0};
static std::atomic<int> g_fail_count{0};

static int cuda_fail(cudaError_t e) {
    t_last_cuda = static_cast<int>(e);
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
    // Largest team (32..4 lanes) that keeps >= 85% of its lanes busy on the last pass over the row;
    // otherwise the best-utilized one.
    int best = 5;
    double best_eff = -1.0;
    for (int l2 = 5; l2 >= 2; --l2) {
        const int L = 1 << l2;
        const double eff = static_cast<double>(units) / (L * ((units + L - 1) / L));
        if (eff >= 0.85) return l2;
        if (eff > best_eff + 1e-9) { best_eff = eff; best = l2; }
    }
    return best;
}

// Tuning override (set through qgemv_tune_override; all zero = planner decides).
static std::atomic<int> g_ovr_threads{0}, g_ovr_l2{-1}, g_ovr_rows{0}, g_ovr_stages{0};

// occ_override > 0 skips the occupancy query (host-only planning for introspection).
//
// Plan.  A warp work item is R whole rows when a row fits in CHUNK_TARGET bytes (R a multiple of the
// 32/L row teams of a warp, sized near CHUNK_TARGET), otherwise one row streamed by the whole warp in
// copies of `chunk_blocks` blocks (whole lane passes of units, near CHUNK_TARGET bytes).  Each warp owns
// a ring of `stages` slots; CTAs have `threads` threads; the grid is persistent (at most SMs x resident
// CTAs).  Small matrices use fewer rows per item so the items spread over the SMs.
static int make_plan(int variant, int m, int N, int K, int sms, unsigned* err, int occ_override, Plan* p) {
    const Geometry g = geometry(variant);
    const int nb = K / g.block_elems;
    const long long rb = static_cast<long long>(nb) * g.block_bytes;
    const int units = nb * g.units_per_block;
    const unsigned xb = x_stage_bytes(variant, m, K);
    constexpr long long CHUNK_TARGET = 2048;

    int l2 = pick_lanes_log2(units);
    int threads = GEMV_THREADS;
    long long R = 1;
    int chunks = 1, chunk_blocks = nb;
    if (rb <= CHUNK_TARGET) {
        // Wider row teams (fewer rows per item) when a full set of teams would overfill an item.
        while (l2 < 5 && (32LL >> l2) * rb > CHUNK_TARGET + CHUNK_TARGET / 2) ++l2;
        const long long teams = 32 >> l2;
        const long long kk = CHUNK_TARGET / (teams * rb);
        R = teams * (kk < 1 ? 1 : kk);
        // Spread: aim for >= 2 work items per warp of a full wave (SMs x 16 warps).
        const long long want = 2LL * sms * 16;
        if ((N + R - 1) / R < want) {
            long long r2 = (N + want - 1) / want;
            r2 = (r2 + teams - 1) / teams * teams;
            if (r2 < R) R = r2;
        }
    } else {
        l2 = 5;
        const int pass = 32 / g.units_per_block;  // blocks per full pass of 32 lanes
        int cb = static_cast<int>(CHUNK_TARGET / g.block_bytes) / pass * pass;
        if (cb < pass) cb = pass;
        chunk_blocks = cb < nb ? cb : nb;
        chunks = (nb + chunk_blocks - 1) / chunk_blocks;
    }
    if (g_ovr_threads.load() > 0) threads = g_ovr_threads.load();
    if (g_ovr_l2.load() >= 0 && chunks == 1) l2 = g_ovr_l2.load();
    if (g_ovr_rows.load() > 0 && chunks == 1) R = g_ovr_rows.load();
    if (R > N) R = N;
    if (R < 1) R = 1;
    const int warps = threads / 32;
    const long long item_bytes = chunks == 1 ? R * rb : static_cast<long long>(chunk_blocks) * g.block_bytes;

    int stages = g_ovr_stages.load() > 0 ? g_ovr_stages.load() : 4;
    if (stages > MAX_STAGES) stages = MAX_STAGES;
    auto need = [&](int s) {
        return BAR_BYTES + xb + static_cast<unsigned long long>(warps) * s * slot_bytes(item_bytes);
    };
    while (stages > 2 && need(stages) > SMEM_CAP) --stages;
    if (need(stages) > SMEM_CAP) return QGEMV_ERR_UNSUPPORTED;

    GemvArgs& a = p->a;
    a.row_bytes = rb;
    a.total_bytes = rb * N;
    a.N = N;
    a.K = K;
    a.rows_per_tile = static_cast<int>(R);
    a.num_tiles = static_cast<int>((N + R - 1) / R);
    a.chunks = chunks;
    a.chunk_blocks = chunk_blocks;
    a.blocks_per_row = nb;
    a.units_per_row = units;
    a.lanes_log2 = l2;
    a.stages = stages;
    a.stage_bytes = slot_bytes(item_bytes);
    a.x_off = BAR_BYTES;
    a.w_off = BAR_BYTES + xb;
    a.err = err;
    p->smem = static_cast<unsigned>(need(stages));
    p->threads = threads;

    int occ = occ_override;
    if (occ < 1) {
        const void* fn = gemv_kernel_ptr(variant, m);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, p->smem) != cudaSuccess || occ < 1)
            occ = 1;
    }
    const long long ctas_needed = (static_cast<long long>(a.num_tiles) + warps - 1) / warps;
    const long long cap = static_cast<long long>(sms) * occ;
    p->grid = static_cast<int>(ctas_needed < cap ? ctas_needed : cap);
    return QGEMV_OK;
}

static int ensure_attr(DeviceInfo& dev, int variant, int m) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev.attr_set[variant][m]) return QGEMV_OK;
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel_ptr(variant, m), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_CAP));
    if (e != cudaSuccess) return cuda_fail(e);
    dev.attr_set[variant][m] = true;
    return QGEMV_OK;
}

cudaError_t launch_gemv(int variant, int m, const GemvArgs& a, int grid, int threads, unsigned smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    GemvArgs copy = a;
    void* args[] = {&copy};
    cudaError_t e = cudaLaunchKernelExC(&cfg, gemv_kernel_ptr(variant, m), args);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

static int run_gemv(int variant, const void* W, const void* x, float* y, int m, int N, int K, void* stream) {
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st) return st;
    if ((st = ensure_attr(*dev, variant, m))) return st;
    const unsigned long long key = (static_cast<unsigned long long>(variant) << 60) |
                                   (static_cast<unsigned long long>(m) << 56) |
                                   (static_cast<unsigned long long>(N) << 28) | static_cast<unsigned long long>(K);
    Plan p;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = dev->plans.find(key);
        if (it != dev->plans.end()) p = it->second;
        else {
            if ((st = make_plan(variant, m, N, K, dev->sms, dev->err, 0, &p))) return st;
            dev->plans.emplace(key, p);
        }
    }
    p.a.W = static_cast<const uint8_t*>(W);
    p.a.x = static_cast<const uint8_t*>(x);
    p.a.y = y;
    cudaError_t e = launch_gemv(variant, m, p.a, p.grid, p.threads, p.smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    g_routes[1 + variant * 8 + (m - 1)].fetch_add(1, std::memory_order_relaxed);
    return QGEMV_OK;
}

static int check_common(int m, int N, int K, int block_elems) {
    if (m < 1 || N < 1 || K < 1) return QGEMV_ERR_INVALID_ARG;
    if (K % block_elems) return QGEMV_ERR_INVALID_ARG;
    if (m > 8) return QGEMV_ERR_UNSUPPORTED;
    return QGEMV_OK;
}

static int variant_of(int fmt) {
    switch (fmt) {
    case QGEMV_Q4_K: return V_Q4K;
    case QGEMV_Q6_K: return V_Q6K;
    case QGEMV_Q8_0: return V_Q80;
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
    const int v = fmt == 4 ? V_W8A16 : variant_of(fmt);
    if (v < 0 || !out || num_sms < 1 || ctas_per_sm < 1) return QGEMV_ERR_INVALID_ARG;
    int st;
    if ((st = check_common(m, N, K, geometry(v).block_elems))) return st;
    if (K > max_k(v, m)) return QGEMV_ERR_UNSUPPORTED;
    Plan p;
    if ((st = make_plan(v, m, N, K, num_sms, nullptr, ctas_per_sm, &p))) return st;
    const long long vals[13] = {1LL << p.a.lanes_log2, p.a.rows_per_tile, p.a.num_tiles, p.a.stages,
                                p.a.stage_bytes, p.smem, p.grid, p.a.row_bytes, p.a.units_per_row,
                                static_cast<long long>(p.a.w_off) - p.a.x_off, p.threads, p.a.chunks,
                                p.a.chunk_blocks};
    for (int i = 0; i < 13; ++i) out[i] = vals[i];
    return QGEMV_OK;
}

void qgemv_tune_override(int threads, int lanes_log2, int rows_per_tile, int stages) {
    g_ovr_threads.store(threads == 128 || threads == 256 ? threads : 0);
    g_ovr_l2.store(lanes_log2 >= 0 && lanes_log2 <= 5 ? lanes_log2 : -1);
    g_ovr_rows.store(rows_per_tile > 0 ? rows_per_tile : 0);
    g_ovr_stages.store(stages >= 2 && stages <= MAX_STAGES ? stages : 0);
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& d : g_dev) d.plans.clear();
}

int qgemv_quantize_act(const float* x, int m, int K, void* xq, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    if ((st = check_common(m, 1, K, 32))) return st;
    if (!x || !xq) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(xq, 16)) return QGEMV_ERR_MISALIGNED;
    if (overlaps(x, static_cast<size_t>(m) * K * 4, xq, qgemv_act_bytes(m, K))) return QGEMV_ERR_OVERLAP;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev))) return st;
    cudaError_t e = launch_quantize(x, m, K, static_cast<uint8_t*>(xq), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    g_routes[0].fetch_add(1, std::memory_order_relaxed);
    return QGEMV_OK;
}

int qgemv(int fmt, const void* W, const void* xq, float* y, int m, int N, int K, void* stream) {
    int st;
    if (take_injected_failure(&st)) return st;
    const int v = variant_of(fmt);
    if (v < 0) return QGEMV_ERR_INVALID_ARG;
    if ((st = check_common(m, N, K, geometry(v).block_elems))) return st;
    if (!W || !xq || !y) return QGEMV_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(y, 4)) return QGEMV_ERR_MISALIGNED;
    if (K > max_k(v, m)) return QGEMV_ERR_UNSUPPORTED;
    const size_t wbytes = qgemv_weight_bytes(fmt, N, K);
    const size_t ybytes = static_cast<size_t>(m) * N * 4;
    if (overlaps(y, ybytes, W, wbytes) || overlaps(y, ybytes, xq, qgemv_act_bytes(m, K))) return QGEMV_ERR_OVERLAP;
    return run_gemv(v, W, xq, y, m, N, K, stream);
}

int qgemv_w8a16(const void* W, const void* x_bf16, float* y, int m, int N, int K, void* stream) {
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
    return run_gemv(V_W8A16, W, x_bf16, y, m, N, K, stream);
}

}  // extern "C"
