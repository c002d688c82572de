// Persistent chained-decode kernel (sm_103a): one cooperative launch runs a list of steps -- GEMVs over one
// or several matrices that share an activation, and activation quantizations -- in order.  Every CTA stays
// resident for the whole chain:
//   - the producer warp streams the weight tiles of step after step into the shared-memory ring without
//     waiting for anything but free slots, so the weights of step i+1 are already in flight while step i
//     finishes;
//   - the consumer warps run each step exactly as the single-launch kernel does (same staging, same decode,
//     same per-row arithmetic, so every output is bit-identical to the one-call result) and then meet the
//     other CTAs at a grid-wide barrier before the next step reads what this one wrote.
// The barrier replaces the end of one launch and the dependency release of the next; with the weights
// prefetched across it, short steps cost about one barrier and one activation staging each.  The decode
// sweep of a transformer (q/k/v, o, gate/up, down per layer, then lm_head) is one such chain, like the
// graph-replayed decode step of vllm.cpp PR #1936 (its HIP graph decode capture section), with the graph
// folded into a single resident launch.
#include "gemv_kernel.cuh"
#include "quantize.cuh"

namespace qg {

static_assert(2 * sizeof(ChainStep) + 64 <= 1024, "the step descriptor copies must fit the static shared reserve");

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier b of the consumer threads of all CTAs (co-resident under the cooperative launch).
// Every barrier has its own arrival counter: a CTA adds 1 with release semantics and polls (acquire) until
// the counter reaches the grid size, for at most WAIT_LIMIT_NS.  Counters go back to zero behind the
// chain: CTA 0 clears counter b - 1 once barrier b is complete (every CTA has then left barrier b - 1), and
// the last CTA to finish clears the last one.  After a wait that ran out the CTA records the error and stops
// waiting at later barriers (its results are then undefined, but the launch still ends).
__device__ __forceinline__ void chain_barrier(const ChainCtl& c, int b, int tid, int NC, bool* alive) {
    consumer_sync(NC * 32);
    if (tid == 0 && *alive) {
        unsigned* cnt = c.bar + CHAIN_BAR_FIRST + b;
        __threadfence();  // this CTA's writes of the finished step before its arrival
        red_release_add(cnt, 1u);
        const unsigned long long t0 = global_ns();
        while (ld_acquire(cnt) < gridDim.x) {
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                atomicOr(c.err, ERR_BARRIER_TIMEOUT);
                *alive = false;
                break;
            }
        }
        if (blockIdx.x == 0 && b > 0 && *alive) atomicExch(cnt - 1, 0u);
    }
    consumer_sync(NC * 32);
}

// End of the chain for one CTA: the last CTA to get here clears the last barrier's counter and the exit count.
__device__ __forceinline__ void chain_exit(const ChainCtl& c, int tid) {
    if (tid == 0 && c.nsteps > 1) {
        __threadfence();
        if (atomicAdd(c.bar + CHAIN_BAR_EXIT, 1u) == gridDim.x - 1) {
            atomicExch(c.bar + CHAIN_BAR_FIRST + (c.nsteps - 2), 0u);
            atomicExch(c.bar + CHAIN_BAR_EXIT, 0u);
        }
    }
}

// One step's descriptor into shared memory, by the consumer threads.
__device__ __forceinline__ void load_step(ChainStep* dst, const ChainStep& st, int tid, int nthreads) {
    for (int w = tid; w < static_cast<int>(sizeof(ChainStep) / 4); w += nthreads)
        reinterpret_cast<uint32_t*>(dst)[w] = reinterpret_cast<const uint32_t*>(&st)[w];
}

template <int V>
__device__ __forceinline__ void chain_gemv(const GemvArgs& a, const Ring& r, uint8_t* xsm, int tid, int warp,
                                           int lane_w, int NC, int& s, uint32_t& fphase) {
    stage_x<V, 1>(a, xsm, tid, NC * 32);
    consumer_sync(NC * 32);
    float bv[1];
    int bn[1];
    consume<V, 1, false>(a, r, xsm, warp, lane_w, NC, s, fphase, bv, bn);
}

__global__ void __launch_bounds__(GEMV_THREADS_MAX, 2) gemv_chain_kernel(const ChainCtl c) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ ChainStep sa[2];  // the current and the next step's descriptors, for the consumers
    __shared__ bool alive;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane_w = tid & 31;
    const int NC = (blockDim.x >> 5) - 1;
    const Ring r = make_ring(smem, c.stages, c.stage_bytes, c.red_off, c.w_off, c.rstride);
    if (tid == 0) alive = true;
    ring_init(r, NC, tid);

    if (warp == NC) {
        // ---------------- producer: every step's tiles, back to back ----------------
        if (lane_w == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int k = 0, s = 0;
            uint32_t ephase = 0;
            bool ok = true;
            for (int i = 0; i < c.nsteps && ok; ++i)
                if (c.steps[i].op == CHAIN_GEMV) ok = produce(c.steps[i].a, r, pol, k, s, ephase);
            if (ok) producer_drain(r, k, c.err);
        }
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();
    uint8_t* xsm = smem + c.x_off;
    int s = 0;
    uint32_t fphase = 0;
    load_step(&sa[0], c.steps[0], tid, NC * 32);
    for (int i = 0; i < c.nsteps; ++i) {
        if (i > 0) chain_barrier(c, i - 1, tid, NC, &alive);  // also publishes sa[i & 1] to every warp
        else consumer_sync(NC * 32);
        const GemvArgs& a = sa[i & 1].a;
        const int op = sa[i & 1].op, variant = sa[i & 1].variant;
        if (op == CHAIN_QUANTIZE) {
            // fp32 [1, K] -> q8_1 over the consumer threads of every CTA, eight lanes per block (the
            // quantizer launch's arithmetic)
            const int nblocks = a.K >> 5;
            const int groups = static_cast<int>(gridDim.x) * NC * 4;  // eight-lane groups in the grid
            const int g = static_cast<int>(blockIdx.x) * NC * 4 + (tid >> 3);
            for (int b0 = 0; b0 < nblocks; b0 += groups)
                quantize_block_part<ACT_F32>(a.x, b0 + g, tid & 7, b0 + g < nblocks, a.xq_out);
        } else {
            switch (variant) {
            case V_Q4K: chain_gemv<V_Q4K>(a, r, xsm, tid, warp, lane_w, NC, s, fphase); break;
            case V_Q5K: chain_gemv<V_Q5K>(a, r, xsm, tid, warp, lane_w, NC, s, fphase); break;
            case V_Q6K: chain_gemv<V_Q6K>(a, r, xsm, tid, warp, lane_w, NC, s, fphase); break;
            default: chain_gemv<V_Q80>(a, r, xsm, tid, warp, lane_w, NC, s, fphase); break;
            }
        }
        // the next step's descriptor, fetched before the barrier so that its latency is off the chain
        if (i + 1 < c.nsteps) load_step(&sa[(i + 1) & 1], c.steps[i + 1], tid, NC * 32);
    }
    chain_exit(c, tid);
}

const void* chain_kernel_ptr() { return reinterpret_cast<const void*>(&gemv_chain_kernel); }

cudaError_t launch_chain(const ChainCtl& c, int grid, int threads, unsigned smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ChainCtl copy = c;
    void* args[] = {&copy};
    cudaError_t e = cudaLaunchKernelExC(&cfg, chain_kernel_ptr(), args);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

}  // namespace qg
