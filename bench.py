#!/usr/bin/env python3
"""Decode-sweep benchmark for libqgemv.

One step = one decode-token sweep of the workload: every activation input quantized once
(qgemv_quantize_act), then every weight matrix streamed once (qgemv / qgemv_w8a16), in layer order.
The metric is effective weight bandwidth: weight bytes of the sweep / sweep time (GB/s), with the
sweep time in microseconds alongside.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Default workload: dense-4b-class (36 layers, hidden 2560, Q4_K/Q6_K projections, Q6_K lm_head, m=1).
Its 2.59 GB of weights exceed twice the L2 cache, so no flush is needed between steps.
The headline replays the whole sweep as one CUDA graph; an eager pass with CUDA events around every
launch gives the per-kernel times used for the roofline.  `--impl reference` times the CPU oracle (the
plain fp64 statement of the method) on a bounded sample of the same workload.
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective weight GB/s (% of GB300 HBM peak) & µs/decode-token sweep, m=1"
FALLBACK_HBM_GBS = 6800.0  # profiling-recipe fallback when no measured peak file exists
# single-row launches of fewer weight bytes than this run the library's register-capped build
SHORT_GEMV_BYTES = 4 << 20
PROFILES = os.path.join(ROOT, "profiles")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="dense-4b-class")
    p.add_argument("--mode", choices=("graph", "eager"), default="graph",
                   help="headline launch mode (graph = one CUDA graph per sweep)")
    p.add_argument("--sweep", choices=("fused", "percall"), default="fused",
                   help="fused: one launch per same-input group with in-kernel quantization; "
                        "percall: a quantize launch per input and a GEMV launch per matrix")
    p.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-all-cores", action="store_true", help="skip the all-cores oracle baseline")
    p.add_argument("--quick", action="store_true", help="skip the instrumented and e2e passes (profiling runs)")
    p.add_argument("--override", default=None,
                   help="force plan parameters ctas_per_sm,lanes_log2,rows_per_tile,stages (-1/0 = planner); "
                        "tuning runs only")
    p.add_argument("--pdl", action="store_true", help="launch with programmatic dependent launch")
    p.add_argument("--pairs", choices=("auto", "on", "off"), default="auto",
                   help="row pairs (two rows per row team) for the builds that have them; tuning runs only")
    p.add_argument("--fuse-max", type=int, default=None,
                   help="fused sweep: activations of at most this many values (m*K) are quantized inside the "
                        "GEMV launch, longer ones by their own quantize launch")
    p.add_argument("--op", default=None,
                   help="single-matrix microbenchmark FMT:N:K[:m] (FMT in Q4_K, Q5_K, Q6_K, Q8_0, W8A16, "
                        "W8A16_CHANNEL); rotates weight copies so that the bytes between reuses exceed twice the "
                        "L2 cache")
    p.add_argument("--timeline", action="store_true",
                   help="run one sweep of the workload on the launch-timeline build of the library and print the "
                        "per-launch breakdown (dependency release, activation staging, tile decode, tail)")
    p.add_argument("--argmax", choices=["fused", "two-pass"], default=None,
                   help="with --op on a K-quant or Q8_0 matrix at m=1: the fused GEMV + argmax launch, or for "
                        "comparison the GEMV followed by torch.argmax over its output")
    return p.parse_args()


# ---------------------------------------------------------------------------------------------------
# peaks, clocks

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBs", "hbm"):
                if key in d:
                    v = d[key]
                    if isinstance(v, dict):
                        v = v.get("burst", v.get("value"))
                    return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """Polls NVML (read-only queries) every ~1 ms from a thread during the timed region: SM clock, max SM
    clock and the clock-event (throttle) reason bits."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        self.dev = device_index
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        self.max_mhz = None

    def _open(self):
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            bus = torch.cuda.get_device_properties(self.dev).pci_bus_id
            ok = nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus.encode()), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.dev), ctypes.byref(h)) != 0:
            return False
        self.nvml, self.handle = nv, h
        mx = ctypes.c_uint(0)
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        return True

    def _sample(self):
        nv, h = self.nvml, self.handle
        c = ctypes.c_uint(0)
        r = ctypes.c_ulonglong(0)
        if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) != 0:
            return None
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        if fn(h, ctypes.byref(r)) != 0:
            r.value = 0
        return c.value, r.value

    def _run(self):
        while not self.stop_flag.is_set():
            v = self._sample()
            if v is not None:
                self.samples.append(v)
            time.sleep(0.001)

    def start(self):
        if not self._open():
            return
        v = self._sample()
        if v is not None:
            self.samples.append(v)
        self.samples = []
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        if self.thread is None:
            return None
        self.stop_flag.set()
        self.thread.join(timeout=2)
        v = self._sample()  # at least one sample at the end of the region
        if v is not None:
            self.samples.append(v)
        if not self.samples:
            return None
        reasons = set()
        for _, bits in self.samples:
            for b, nm in self.REASONS.items():
                if bits & b:
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml"}


# ---------------------------------------------------------------------------------------------------
# the sweep on the GPU

class Sweep:
    """Device-resident weights, activations and outputs of one workload, and its launch lists.

    Two ways to issue one decode-token sweep through the library:
      fused   - one qgemv_multi launch per group of consecutive matrices that read the same input (e.g.
                q/k/v, gate/up); short fp32 activations are quantized inside that launch, longer ones by
                one quantize launch before it;
      percall - one qgemv_quantize_act per distinct input, then one qgemv per matrix.
    Both use programmatic dependent launch between consecutive library kernels when `pdl` is set.
    """

    # Fused sweep: activations of at most this many values are quantized inside the GEMV launch.  Every CTA
    # of the launch quantizes the whole row, which costs more than one quantize launch once the row is
    # longer than a few thousand values.
    FUSE_MAX_DEFAULT = 2048

    def _layout(self, wl, qg):
        """Byte offsets of every weight matrix, activation, quantized activation and output in the sweep's
        buffers (host only): sets offs, inputs, xq, youts, w8 and returns the four buffer sizes."""
        m = wl.m
        # weights: one allocation, each matrix 256-byte aligned
        self.offs, total = [], 0
        for g in wl.gemvs:
            self.offs.append(total)
            total += (g.weight_bytes + 255) // 256 * 256
        # activations: one contiguous fp32 (or bf16 for W8A16) buffer, each input 256-byte aligned
        self.inputs = {}
        in_bytes = 0
        self.w8 = any(g.w8a16 for g in wl.gemvs)
        esize = 2 if self.w8 else 4
        for name, K in wl.inputs():
            self.inputs[name] = (in_bytes, K)
            in_bytes += (m * K * esize + 255) // 256 * 256
        # quantized activations (percall mode)
        self.xq = {}
        q_total = 0
        for name, (o, K) in self.inputs.items():
            self.xq[name] = q_total
            q_total += (qg.qgemv_act_bytes(m, K) + 255) // 256 * 256
        # outputs: one contiguous buffer
        self.youts, y_total = [], 0
        for g in wl.gemvs:
            self.youts.append(y_total)
            y_total += (m * g.N * 4 + 255) // 256 * 256
        return total, in_bytes, max(q_total, 256), y_total

    def __init__(self, wl, torch, qg, gen, fuse_max=None):
        from qgemv_inputs import workloads as W
        self.fuse_max = self.FUSE_MAX_DEFAULT if fuse_max is None else fuse_max
        self.wl = wl
        self.torch = torch
        self.qg = qg
        self.L = qg.lib()
        m = wl.m
        dev = torch.device("cuda")
        total, in_bytes, q_total, y_total = self._layout(wl, qg)
        offs = self.offs
        esize = 2 if self.w8 else 4
        self.wbuf = torch.empty(total, dtype=torch.uint8, device=dev)
        for g, o in zip(wl.gemvs, offs):
            host = gen.weights(g.fmt, g.N, g.K, W.weight_seed(wl, g))
            self.wbuf[o:o + g.weight_bytes].copy_(torch.from_numpy(host))
        self.h_in = torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True)
        hv = self.h_in.numpy()
        for name, (o, K) in self.inputs.items():
            for i in range(m):
                seed = W.input_seed(wl, name, i)
                row = gen.normal_bf16(K, seed).view("u1") if self.w8 else gen.normal_f32(K, seed).view("u1")
                hv[o + i * K * esize:o + (i + 1) * K * esize] = row
        self.d_in = self.h_in.to(dev)
        self.d_xq = torch.empty(q_total, dtype=torch.uint8, device=dev)
        self.d_out = torch.empty(y_total, dtype=torch.uint8, device=dev)
        # the step's result, read back by the end-to-end pass: the last launch's output (the lm_head's logits;
        # the other outputs stand for activations a model keeps on the device)
        last = wl.gemvs[-1]
        self.result_off, self.result_bytes = self.youts[-1], m * last.N * 4
        self.h_out = torch.empty(self.result_bytes, dtype=torch.uint8, pin_memory=True)
        self.weight_bytes = wl.weight_bytes

    def calls(self, mode, pdl):
        """[(kernel key, fn, args without stream, algorithmic bytes, keepalive)] for one sweep."""
        from qgemv_inputs import workloads as W
        qg, L, wl, m = self.qg, self.L, self.wl, self.wl.m
        flags = qg.QGEMV_FLAG_PDL if pdl else 0

        def quant_flags(f, next_weight_bytes):
            # a quantize launch before a short GEMV (the library's register-capped single-row build, below
            # 4 MB of weights) lets it start only after its own dependency wait: measured faster there
            # (0.6B-class sweep 433.6 -> 411.3 us) and slower before long GEMVs
            if f & qg.QGEMV_FLAG_PDL and m == 1 and next_weight_bytes < SHORT_GEMV_BYTES:
                return f | qg.QGEMV_FLAG_PDL_LATE_TRIGGER
            return f
        wp, ip, qp, yp = self.wbuf.data_ptr(), self.d_in.data_ptr(), self.d_xq.data_ptr(), self.d_out.data_ptr()
        out = []
        gemvs = list(enumerate(wl.gemvs))
        if mode == "percall":
            gi = 0
            for j, op in enumerate(wl.ops):
                if isinstance(op, W.QuantOp):
                    o, K = self.inputs[op.input]
                    nxt = next((g for g in wl.ops[j + 1:] if not isinstance(g, W.QuantOp)), None)
                    qf = quant_flags(flags, nxt.weight_bytes if nxt is not None else 0)
                    out.append(("quantize", L.qgemv_quantize_act_ex, (ip + o, m, K, qp + self.xq[op.input], qf),
                                m * K * 4 + qg.qgemv_act_bytes(m, K), None))
                    continue
                g = op
                o, K = self.inputs[g.input]
                y = yp + self.youts[gi]
                if g.w8a16:
                    out.append((f"W8A16/m{m}", L.qgemv_w8a16_ex, (wp + self.offs[gi], ip + o, y, m, g.N, g.K, flags),
                                g.weight_bytes + m * K * 2 + m * g.N * 4, None))
                else:
                    out.append((f"{g.fmt}/m{m}", L.qgemv_ex,
                                (qg.FMT[g.fmt], wp + self.offs[gi], qp + self.xq[g.input], y, m, g.N, g.K, flags),
                                g.weight_bytes + qg.qgemv_act_bytes(m, K) + m * g.N * 4, None))
                gi += 1
            return out
        # fused: consecutive matrices with the same input and format form one launch.  A short
        # activation (m*K <= fuse_max values) is quantized inside that launch; a longer one is quantized
        # once by its own launch.
        FUSE_MAX = self.fuse_max
        groups = []
        for gi, g in gemvs:
            if groups and groups[-1][0].input == g.input and groups[-1][0].fmt == g.fmt and \
                    groups[-1][0].w8a16 == g.w8a16 and len(groups[-1][1]) < qg.QGEMV_MAX_GROUP:
                groups[-1][1].append(gi)
            else:
                groups.append((g, [gi]))
        for g0, idx in groups:
            o, K = self.inputs[g0.input]
            mats = qg.mats_array([(wp + self.offs[i], yp + self.youts[i], wl.gemvs[i].N) for i in idx])
            wbytes = sum(wl.gemvs[i].weight_bytes for i in idx)
            ybytes = sum(m * wl.gemvs[i].N * 4 for i in idx)
            if g0.w8a16:
                out.append((f"W8A16/m{m}", L.qgemv_multi,
                            (qg.QGEMV_W8A16, len(idx), mats, qg.QGEMV_ACT_BF16, ip + o, None, m, K, flags),
                            wbytes + m * K * 2 + ybytes, mats))
            elif m * K <= FUSE_MAX:
                out.append((f"{g0.fmt}/m{m}", L.qgemv_multi,
                            (qg.FMT[g0.fmt], len(idx), mats, qg.QGEMV_ACT_F32, ip + o, None, m, K, flags),
                            wbytes + m * K * 4 + ybytes, mats))
            else:
                xq = qp + self.xq[g0.input]
                out.append(("quantize", L.qgemv_quantize_act_ex, (ip + o, m, K, xq, quant_flags(flags, wbytes)),
                            m * K * 4 + qg.qgemv_act_bytes(m, K), None))
                out.append((f"{g0.fmt}/m{m}", L.qgemv_multi,
                            (qg.FMT[g0.fmt], len(idx), mats, qg.QGEMV_ACT_Q8_1, xq, None, m, K, flags),
                            wbytes + qg.qgemv_act_bytes(m, K) + ybytes, mats))
        return out

    @staticmethod
    def run(calls, stream_handle):
        s = ctypes.c_void_p(stream_handle)
        for key, fn, args, _, _ in calls:
            st = fn(*args, s)
            if st != 0:
                raise RuntimeError(f"{key}: status {st}")


def max_over_ranks(ms, dist, device):
    """The slowest rank's time per step (every rank gets it); `dist` None means one process."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sweep_value(world, weight_bytes, ms):
    """Whole-job effective weight GB/s: every rank sweeps the full weight set once per step."""
    return world * weight_bytes / (ms * 1e-3) / 1e9


def _graph_of(torch, calls, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            Sweep.run(calls, stream.cuda_stream)
    return g


def _time_graph(torch, g, stream, reps):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / reps


def kernel_launches(qg, run, stream):
    """Kernels one pass of `run` launches, from the library's route counters: the quantizer and one count
    per GEMV launch (a call the library serves as two launches counts twice); the attribute counters
    (in-kernel quantization, grouped, PDL, argmax) are not launches of their own."""
    stream.synchronize()
    qg.qgemv_route_reset()
    run()
    stream.synchronize()
    c = qg.qgemv_route_counts()
    attrs = {qg.ROUTE_FUSED, qg.ROUTE_GROUPED, qg.ROUTE_PDL, qg.ROUTE_ARGMAX, qg.ROUTE_CHUNKED}
    return sum(v for i, v in enumerate(c) if i not in attrs)


def run_ours(args, rank, world, local_rank):
    import torch
    import qgemv_inputs as gen
    import quantized_weight_gemv_quantize_gb300 as qg
    from qgemv_inputs.workloads import WORKLOADS
    import __graft_entry__

    torch.cuda.set_device(local_rank)
    __graft_entry__.build()
    wl = WORKLOADS[args.workload]()
    if args.override:
        qg.qgemv_tune_override(*(int(v) for v in args.override.split(",")))
    qg.qgemv_tune_pairs({"auto": 0, "on": 1, "off": 2}[args.pairs])
    sw = Sweep(wl, torch, qg, gen, args.fuse_max)
    stream = torch.cuda.Stream()
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    pdl = not args.no_pdl
    calls = sw.calls(args.sweep, pdl)
    # warm-up (also initializes the library's per-device state before any capture)
    for _ in range(max(args.warmup, 1)):
        Sweep.run(calls, stream.cuda_stream)
    stream.synchronize()
    n_launch = kernel_launches(qg, lambda: Sweep.run(calls, stream.cuda_stream), stream)
    graph = None
    if args.mode == "graph":
        graph = _graph_of(torch, calls, stream)
        for _ in range(args.warmup):
            with torch.cuda.stream(stream):
                graph.replay()
        stream.synchronize()

    def step():
        if graph is not None:
            with torch.cuda.stream(stream):
                graph.replay()
        else:
            Sweep.run(calls, stream.cuda_stream)

    # Weights that fit twice in L2 would be served from L2 by the next step: then every step is timed on
    # its own and a buffer larger than L2 is written between steps (outside the timed spans).
    l2_bytes = torch.cuda.get_device_properties(local_rank).L2_cache_size
    flush = sw.weight_bytes < 2 * l2_bytes
    scrub = torch.empty(2 * l2_bytes, dtype=torch.uint8, device="cuda") if flush else None
    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    def timed_round():
        """ms per step over K steps (each step alone, L2 scrubbed before it, when the weights fit in L2)."""
        if flush:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for a, b in evs:
                with torch.cuda.stream(stream):
                    scrub.fill_(1)
                a.record(stream)
                step()
                b.record(stream)
            barrier()
            return sum(a.elapsed_time(b) for a, b in evs) / args.steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / args.steps

    step_ms = timed_round()
    ms = max_over_ranks(step_ms, dist, "cuda")
    # More rounds of K steps for the spread (median / min / max); the headline is the round above.  They
    # run for about two seconds (at least five rounds) so that the clock samples cover a sustained load.
    # The count follows from the headline time, which every rank shares (max over ranks).
    n_rounds = 0 if args.quick else min(500, max(5, int(2.0 / max(ms * 1e-3 * args.steps, 1e-6)) + 1))
    rounds = [max_over_ranks(timed_round(), dist, "cuda") for _ in range(n_rounds)]
    clk = clocks.stop()
    result = {"ms": ms, "clocks": clk, "launches_per_step": n_launch, "pdl": pdl, "sweep": args.sweep, "l2_flush": flush,
              "rounds": rounds,
              "fuse_max": sw.fuse_max}

    if not args.quick:
        reps = max(3, args.steps)
        # the other way of issuing the sweep, for reference
        other = "percall" if args.sweep == "fused" else "fused"
        other_calls = sw.calls(other, pdl)
        Sweep.run(other_calls, stream.cuda_stream)
        result["other"] = {"sweep": other,
                           "launches": kernel_launches(qg, lambda: Sweep.run(other_calls, stream.cuda_stream), stream),
                           "ms": _time_graph(torch, _graph_of(torch, other_calls, stream), stream, reps)}
        # per kernel class: a graph of that class's launches alone (same order, arguments and flags)
        per = {}
        for key in sorted({c[0] for c in calls}):
            sub = [c for c in calls if c[0] == key]
            gms = _time_graph(torch, _graph_of(torch, sub, stream), stream, reps)
            per[key] = {"launches": kernel_launches(qg, lambda: Sweep.run(sub, stream.cuda_stream), stream), "ms": gms,
                        "bytes": sum(c[3] for c in sub)}
        result["kernels"] = per

    if flush and not args.quick:
        # Kernel time of a workload that fits in L2: one graph of sweeps over rotating copies of its weights
        # (every copy once per replay, the copies together more than twice the L2 cache), so each launch
        # reads cold weights, without the scrub and replay overhead of the per-step timing above.
        copies = max(2, -(-2 * l2_bytes // max(1, sw.wbuf.numel())) + 1)
        base = sw.wbuf
        rot = torch.empty((copies, base.numel()), dtype=torch.uint8, device="cuda")
        rot.copy_(base.unsqueeze(0).expand(copies, -1))
        rot_calls = []
        for c in range(copies):
            sw.wbuf = rot[c]
            rot_calls += sw.calls(args.sweep, pdl)
        sw.wbuf = base
        Sweep.run(rot_calls, stream.cuda_stream)
        rot_ms = _time_graph(torch, _graph_of(torch, rot_calls, stream), stream, 3)
        result["kernel_only"] = {"copies": copies, "sweeps_per_graph": copies,
                                 "launches_per_graph": copies * n_launch, "ms_per_sweep": rot_ms / copies}
        del rot

    # end to end: host input -> device, sweep, device output -> host, every step
    if not args.no_e2e and not args.quick:
        d_result = sw.d_out[sw.result_off:sw.result_off + sw.result_bytes]

        def e2e_copies_and_sweep():
            sw.d_in.copy_(sw.h_in, non_blocking=True)
            step()
            sw.h_out.copy_(d_result, non_blocking=True)

        # one graph a step (the inputs' copy in, the sweep, the result's copy back) when the sweep runs as a
        # graph: one launch per token instead of three; the copies stay plain stream copies if capture fails
        e2e_graph = None
        if graph is not None:
            try:
                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    with torch.cuda.graph(g2, stream=stream, capture_error_mode="thread_local"):
                        sw.d_in.copy_(sw.h_in, non_blocking=True)
                        Sweep.run(calls, stream.cuda_stream)
                        sw.h_out.copy_(d_result, non_blocking=True)
                e2e_graph = g2
            except RuntimeError as e:
                result["e2e_graph"] = f"not captured: {type(e).__name__}: {e}"[:200]
                torch.cuda.synchronize()
        result.setdefault("e2e_graph", "captured" if e2e_graph is not None else "no sweep graph")

        def e2e_step():
            with torch.cuda.stream(stream):
                if e2e_graph is not None:
                    e2e_graph.replay()
                else:
                    e2e_copies_and_sweep()
            stream.synchronize()
        for _ in range(args.warmup):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        barrier()
        result["e2e_wall_ms"] = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.steps, dist, "cuda")
        result["e2e_ms"] = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, "cuda")
        result["h2d"] = int(sw.d_in.numel())
        result["d2h"] = int(sw.result_bytes)
    result["weight_bytes"] = sw.weight_bytes
    result["m"] = wl.m
    result["device_error"] = qg.qgemv_device_error()
    return result


# ---------------------------------------------------------------------------------------------------
# the oracle on the host (CPU baseline and the reference arm)

class OracleSample:
    """A bounded sample of the workload for the CPU oracle: the first `frac` of every matrix's rows,
    plus every activation quantization.  Throughput is scaled by weight bytes actually processed."""

    def __init__(self, wl):
        import numpy as np
        import qgemv_inputs as gen
        from qgemv_inputs import workloads as W
        self.np = np
        self.wl = wl
        self.items = []
        xs = {}
        for name, K in wl.inputs():
            w8 = any(g.w8a16 and g.input == name for g in wl.gemvs)
            rows = [gen.normal_bf16(K, W.input_seed(wl, name, i)) if w8 else gen.normal_f32(K, W.input_seed(wl, name, i))
                    for i in range(wl.m)]
            xs[name] = (np.stack(rows), w8)
        self.xs = xs
        self.mats = {}
        for g in wl.gemvs:
            self.mats[g.name] = g

    def run(self, frac):
        import oracle
        import qgemv_inputs as gen
        from qgemv_inputs import workloads as W
        np = self.np
        done = 0
        xq = {}
        for name, (x, w8) in self.xs.items():
            if not w8:
                xq[name] = oracle.quantize_act(x)
        for g in self.wl.gemvs:
            rows = max(1, int(round(g.N * frac)))
            Wfull = self._rows(g, rows)
            x, w8 = self.xs[g.input]
            if w8:
                oracle.w8a16(Wfull, x, self.wl.m, rows, g.K)
            else:
                oracle.gemv(g.fmt, Wfull, xq[g.input], self.wl.m, rows, g.K)
            done += g.weight_bytes * rows // g.N
        return done

    def _rows(self, g, rows):
        import qgemv_inputs as gen
        from qgemv_inputs import workloads as W
        key = (g.name, rows)
        if not hasattr(self, "_cache"):
            self._cache = {}
        if key not in self._cache:
            # the first `rows` rows of the matrix are the first rows*K/blk blocks of its stream
            self._cache[key] = gen.weights(g.fmt, rows, g.K, W.weight_seed(self.wl, g))
        return self._cache[key]


def oracle_throughput(wl, seconds_target):
    s = OracleSample(wl)
    frac = 1.0 / 4096
    while True:
        t0 = time.perf_counter()
        b = s.run(frac)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * seconds_target or frac >= 1.0:
            return b, dt, frac, s
        frac = min(1.0, frac * min(64.0, seconds_target / max(dt, 1e-3)))


_ORACLE_BARRIER = None


def _oracle_worker_init(barrier):
    global _ORACLE_BARRIER
    _ORACLE_BARRIER = barrier


def _oracle_worker(task):
    """One process of the all-cores oracle baseline: one warm pass over the bounded sample, then every
    process starts its timed pass together (a barrier) so that the passes overlap."""
    name, frac = task
    from qgemv_inputs.workloads import WORKLOADS
    s = OracleSample(WORKLOADS[name]())
    s.run(frac)
    _ORACLE_BARRIER.wait(timeout=300)
    t0 = time.perf_counter()
    b = s.run(frac)
    return b, time.perf_counter() - t0


def oracle_all_cores(wl, frac_single):
    """The oracle on every host core: P spawned processes each run the bounded sample (1/P of the
    single-thread sample) at the same time; throughput = all bytes / the slowest process's time."""
    import multiprocessing as mp
    procs = max(1, min(os.cpu_count() or 1, 16))
    frac = max(1.0 / 4096, frac_single / procs)
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(procs)
    with ctx.Pool(procs, initializer=_oracle_worker_init, initargs=(barrier,)) as pool:
        res = pool.map_async(_oracle_worker, [(wl.name, frac)] * procs).get(timeout=600)
    return sum(r[0] for r in res), max(r[1] for r in res), procs, frac


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from qgemv_inputs.workloads import WORKLOADS
    import oracle._build as ob
    import qgemv_inputs._build as gb
    # the oracle arm needs only the oracle and the input generator, never the CUDA library
    gb.build()
    ob.build()
    wl = WORKLOADS[args.workload]()
    # one step = a bounded sample sized so that warmup + steps finish in about two minutes
    per_step = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    _, _, frac, s = oracle_throughput(wl, per_step)
    for _ in range(args.warmup):
        s.run(frac)
    t0 = time.perf_counter()
    tot = 0
    for _ in range(args.steps):
        tot += s.run(frac)
    dt = time.perf_counter() - t0
    gbs = tot / dt / 1e9
    ms_full = wl.weight_bytes / (tot / dt) * 1e3
    sample = f"first {frac:.5f} of every matrix's rows + all activation quantizations, per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_full, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "m": wl.m, "weight_bytes": wl.weight_bytes},
        "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    return line


# ---------------------------------------------------------------------------------------------------

def run_op(args):
    """One GEMV shape, launched `steps` times back to back over rotating weight copies."""
    import numpy as np
    import torch
    import qgemv_inputs as gen
    import quantized_weight_gemv_quantize_gb300 as qg
    import __graft_entry__

    __graft_entry__.build()
    parts = args.op.split(":")
    fmt, N, K = parts[0], int(parts[1]), int(parts[2])
    m = int(parts[3]) if len(parts) > 3 else 1
    w8 = fmt == "W8A16"
    w8c = fmt == "W8A16_CHANNEL"
    wfmt = "Q8_0" if w8 else fmt
    wb = N * K + 4 * N if w8c else qg.qgemv_weight_bytes(wfmt, N, K)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    copies = max(2, -(-2 * l2 // wb) + 1)
    stride = (wb + 255) // 256 * 256
    W = torch.empty(copies * stride, dtype=torch.uint8, device="cuda")
    if w8c:
        wq, sc = gen.channel_weights(N, K, 7)
        host = torch.from_numpy(np.concatenate([wq.view(np.uint8), sc.view(np.uint8)]))
    else:
        host = torch.from_numpy(gen.weights(wfmt, N, K, 7))
    for c in range(copies):
        W[c * stride:c * stride + wb].copy_(host)
    y = torch.empty(m * N, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    if args.override:
        qg.qgemv_tune_override(*(int(v) for v in args.override.split(",")))
    qg.qgemv_tune_pairs({"auto": 0, "on": 1, "off": 2}[args.pairs])
    if w8 or w8c:
        x = torch.from_numpy(np.stack([gen.normal_bf16(K, 3 + i) for i in range(m)])).cuda()
        flags = qg.QGEMV_FLAG_PDL if args.pdl else 0
        if w8c:  # int8 rows, then the fp32 scales, in each copy
            launch = lambda c: qg.qgemv_w8a16_channel(W.data_ptr() + c * stride, W.data_ptr() + c * stride + N * K,
                                                      x, y, m, N, K, flags, stream=stream)
        else:
            launch = lambda c: qg.qgemv_w8a16_ex(W.data_ptr() + c * stride, x, y, m, N, K, flags, stream=stream)
    else:
        x = torch.from_numpy(np.stack([gen.normal_f32(K, 3 + i) for i in range(m)])).cuda()
        xq = torch.empty(qg.qgemv_act_bytes(m, K), dtype=torch.uint8, device="cuda")
        qg.qgemv_quantize_act(x, m, K, xq, stream=stream)
        flags = qg.QGEMV_FLAG_PDL if args.pdl else 0
        if args.argmax == "two-pass":
            def launch(c):
                qg.qgemv_ex(fmt, W.data_ptr() + c * stride, xq, y, m, N, K, flags, stream=stream)
                with torch.cuda.stream(stream):
                    torch.argmax(y)
        elif args.argmax == "fused":
            scratch = torch.zeros(qg.qgemv_argmax_scratch_bytes(m), dtype=torch.uint8, device="cuda")
            idx = torch.empty(m, dtype=torch.int32, device="cuda")
            launch = lambda c: qg.qgemv_argmax(fmt, W.data_ptr() + c * stride, xq, m, N, K, scratch, idx, y, flags,
                                               stream=stream)
        else:
            launch = lambda c: qg.qgemv_ex(fmt, W.data_ptr() + c * stride, xq, y, m, N, K, flags, stream=stream)
    for i in range(args.warmup):
        launch(i % copies)
    stream.synchronize()
    # one CUDA graph holding `steps` launches over the rotating copies: no host time between kernels
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for i in range(args.steps):
                launch(i % copies)
        graph.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        graph.replay()
    e1.record(stream)
    stream.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    peak, kind = hbm_peak()
    plan = qg.qgemv_plan_info("W8A16" if w8 else fmt, m, N, K,
                              num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    print(json.dumps({"op": args.op, "argmax": args.argmax, "override": args.override, "pdl": args.pdl, "us_per_op": round(us, 3), "weight_bytes": wb, "copies": copies,
                      "GBps": round(wb / (us * 1e-6) / 1e9, 1), "frac_of_peak": round(wb / (us * 1e-6) / 1e9 / peak, 4),
                      "peak_kind": kind, "plan": plan, "device_error": qg.qgemv_device_error()}), flush=True)


def run_timeline(args):
    """Per-launch timeline of one graph-replayed sweep on the traced library (libqgemv_trace.so).  Each launch
    is itemized from its CTAs' %globaltimer stamps; times in microseconds:
      release  previous launch's last CTA done -> this launch's first consumer released
      staging  median over CTAs of release -> activation staged
      wait0    median over CTAs of staged -> first tile's slot full (consumer warp 0)
      tile     median over CTAs of one tile's decode (consumer warp 0, first tile)
      run      last CTA staged -> last CTA done
      tail     first CTA done -> last CTA done
      span     previous launch's last CTA done -> this launch's last CTA done
    Stamping adds a few instructions per CTA and tile, so the traced sweep runs a little slower."""
    import numpy as np
    import torch
    import qgemv_inputs as gen
    import quantized_weight_gemv_quantize_gb300 as qg
    import qgemv_inputs._build as gb
    from qgemv_inputs.workloads import WORKLOADS

    gb.build()
    qg.use_trace_build()
    torch.cuda.set_device(0)
    wl = WORKLOADS[args.workload]()
    sw = Sweep(wl, torch, qg, gen, args.fuse_max)
    stream = torch.cuda.Stream()
    calls = sw.calls(args.sweep, not args.no_pdl)
    for _ in range(max(3, args.warmup)):
        Sweep.run(calls, stream.cuda_stream)
    stream.synchronize()
    qg.trace_begin()
    graph = _graph_of(torch, calls, stream)
    for _ in range(max(3, args.warmup)):
        with torch.cuda.stream(stream):
            graph.replay()
    ms = _time_graph(torch, graph, stream, max(3, args.steps))
    tr, n = qg.trace_read()
    tr = tr.astype(np.int64)
    keys = [c[0] for c in calls]
    rows = []
    prev_end = None
    for l in range(min(n, len(calls))):
        e = tr[l][tr[l][:, 7] != 0]
        if len(e) == 0 or keys[l] in ("",):
            prev_end = None
            continue
        end, first_end = int(e[:, 3].max()), int(e[:, 3].min())
        r = {"i": l, "kernel": keys[l], "bytes": calls[l][3], "ctas": len(e),
             "staging": float(np.median(e[:, 2] - e[:, 1])) / 1e3,
             "run": (end - int(e[:, 2].max())) / 1e3, "tail": (end - first_end) / 1e3,
             "tiles_max": int(((e[:, 8] > 0).astype(int) + (e[:, 10] > 0) + (e[:, 12] > 0)).max())}
        if (e[:, 8] > 0).any():
            g = e[e[:, 8] > 0]
            r["wait0"] = float(np.median(g[:, 8] - g[:, 2])) / 1e3
            r["tile"] = float(np.median(g[:, 9] - g[:, 8])) / 1e3
        if prev_end is not None:
            r["release"] = (int(e[:, 1].min()) - prev_end) / 1e3
            r["span"] = (end - prev_end) / 1e3
        prev_end = end
        rows.append(r)
    full = [r for r in rows if "span" in r]
    peak, peak_kind = hbm_peak()
    classes = {}
    for r in full:
        c = classes.setdefault(r["kernel"], {"launches": 0, "bytes": 0, "span_us": 0.0, **{k: 0.0 for k in (
            "release", "staging", "wait0", "tile", "run", "tail")}})
        c["launches"] += 1
        c["bytes"] += r["bytes"]
        c["span_us"] += r["span"]
        for k in ("release", "staging", "wait0", "tile", "run", "tail"):
            c[k] += r.get(k, 0.0)
    print(f"| class | launches | mean release | mean staging | mean wait0 | mean tile | mean run | mean tail | "
          f"mean span | sum of spans (us) | GB/s over spans |")
    print("|---|---|---|---|---|---|---|---|---|---|---|")
    for k, c in sorted(classes.items()):
        nl = c["launches"]
        print(f"| {k} | {nl} | " + " | ".join(f"{c[f] / nl:.2f}" for f in ("release", "staging", "wait0", "tile", "run",
                                                                        "tail", "span_us"))
              + f" | {c['span_us']:.1f} | {c['bytes'] / (c['span_us'] * 1e-6) / 1e9:.0f} |")
    mid = len(full) // 2
    while mid > 0 and full[mid]["kernel"] == full[mid - 1]["kernel"]:
        mid -= 1
    print("\n| launch | kernel | bytes | CTAs | max tiles/CTA | release | staging | wait0 | tile | run | tail | span |")
    print("|---|---|---|---|---|---|---|---|---|---|---|---|")
    for r in full[mid:mid + 8]:
        print(f"| {r['i']} | {r['kernel']} | {r['bytes']} | {r['ctas']} | {r['tiles_max']} | "
              + " | ".join(f"{r.get(k, 0.0):.2f}" for k in ("release", "staging", "wait0", "tile", "run", "tail",
                                                           "span")) + " |")
    print(json.dumps({"timeline": args.workload, "traced_us_per_sweep": round(ms * 1e3, 2), "launches": len(calls),
                      "recorded": len(full), "sum_span_us": round(sum(r["span"] for r in full), 1),
                      "weight_bytes": sw.weight_bytes, "peak_gbs": peak, "peak_kind": peak_kind,
                      "classes": {k: {f: (round(v, 3) if isinstance(v, float) else v) for f, v in c.items()}
                                  for k, c in classes.items()},
                      "device_error": qg.qgemv_device_error()}), flush=True)


def _without_trace_blocks(text):
    """Source lines the product build compiles: `#ifdef QGEMV_TRACE` blocks dropped, their `#else` parts kept
    (the trace blocks are not nested)."""
    out, state = [], None  # state: None outside a trace block, "if" / "else" inside one
    for line in text.split("\n"):
        t = line.strip()
        if state is None and t.startswith("#ifdef QGEMV_TRACE"):
            state = "if"
        elif state is not None and t.startswith("#else"):
            state = "else"
        elif state is not None and t.startswith("#endif"):
            state = None
        elif state in (None, "else"):
            out.append(line)
    return "\n".join(out)


def kernel_source_hash():
    """Hash of the CUDA sources and the header they include as the product library compiles them: comments,
    blank space and the timeline build's QGEMV_TRACE blocks removed.  Traffic figures taken from an ncu
    capture of another build of the kernels do not describe this one."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_weight_gemv_quantize_gb300", "csrc")
    files = [os.path.join(csrc, n) for n in sorted(os.listdir(csrc)) if n.endswith((".cu", ".cuh", ".h"))]
    for f in files + [os.path.join(ROOT, "include", "qgemv.h")]:
        with open(f) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = _without_trace_blocks(text)
        h.update(os.path.basename(f).encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:12]


def traffic_from_profiles(workload, kernel_key):
    """DRAM bytes (read + write) per launch from an ncu capture of the same kernel class, workload and
    source build (profiles/traffic.md rows: | workload | kernel | bytes per launch | source hash | ...)."""
    path = os.path.join(PROFILES, "traffic.md")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    for ln in open(path):
        parts = [p.strip().strip("`") for p in ln.strip().strip("|").split("|")]
        if len(parts) >= 4 and parts[0] == workload and parts[1] == kernel_key and parts[3] == src:
            try:
                return float(parts[2])
            except ValueError:
                return None
    return None


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.timeline:
        run_timeline(args)
        return
    if args.op:
        run_op(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = hbm_peak()
    wb = res["weight_bytes"]
    ms = res["ms"]
    value = sweep_value(world, wb, ms)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "us_per_sweep": round(ms * 1e3, 2),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2), "peak_kind": peak_kind,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8xs8->s32, f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "m": res["m"], "weight_bytes": wb, "launch": args.mode,
                   "sweep": res["sweep"], "pdl": res["pdl"], "fuse_max": res.get("fuse_max"), "launches_per_sweep": res["launches_per_step"],
                   "l2": ("weights fit in L2: a 2x-L2 buffer written between steps, each step timed alone"
                          if res.get("l2_flush") else "sweep weights exceed 2x L2; no flush between steps"),
                   "parallelism": f"replicas{world}", "override": args.override, "pairs": args.pairs},
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": res["clocks"],
    }
    if "other" in res:
        o = res["other"]
        line["other_sweep"] = {"sweep": o["sweep"], "launches_per_sweep": o["launches"],
                               "us_per_sweep": round(o["ms"] * 1e3, 2),
                               "value": round(wb / (o["ms"] * 1e-3) / 1e9, 2)}
    if res.get("rounds"):
        r = sorted(res["rounds"])
        line["rounds"] = {"n": len(r), "steps_each": args.steps, "median_us": round(statistics.median(r) * 1e3, 2),
                          "min_us": round(r[0] * 1e3, 2), "max_us": round(r[-1] * 1e3, 2)}
    if "kernels" in res:
        per = res["kernels"]
        tot = sum(d["ms"] for d in per.values())
        kern = {}
        for k, d in per.items():
            kern[k] = {"launches_per_step": d["launches"], "share": round(d["ms"] / tot, 4),
                       "avg_us": round(1e3 * d["ms"] / d["launches"], 3),
                       "GBps": round(d["bytes"] / (d["ms"] * 1e-3) / 1e9, 1)}
        line["kernels"] = kern
        dom = max((k for k in per if k != "quantize"), key=lambda k: per[k]["ms"])
        d = per[dom]
        achieved = d["bytes"] / (d["ms"] * 1e-3) / 1e9
        traffic = traffic_from_profiles(args.workload, dom)
        line["roofline"] = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                            "unit": "GB/s", "frac": round(achieved / peak, 4),
                            "traffic": traffic, "peak_kind": f"of {peak_kind}",
                            "algorithmic_bytes_per_launch": d["bytes"] // d["launches"]}
    if "kernel_only" in res:
        ko = res["kernel_only"]
        line["kernel_only"] = {"us_per_sweep": round(ko["ms_per_sweep"] * 1e3, 3),
                               "value": round(wb / (ko["ms_per_sweep"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                               "how": f"one CUDA graph of {ko['sweeps_per_graph']} sweeps over as many rotating "
                                      f"weight copies ({ko['launches_per_graph']} launches), cold weights each launch"}
    if "e2e_ms" in res:
        line["e2e"] = {"value": round(sweep_value(world, wb, res["e2e_ms"]), 2), "unit": "GB/s",
                       "ms_per_step": round(res["e2e_ms"], 5), "wall_ms_per_step": round(res["e2e_wall_ms"], 5),
                       "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                       "launch": res.get("e2e_graph", "")}
    if world == 1 and not args.no_cpu_baseline:
        from qgemv_inputs.workloads import WORKLOADS
        wl = WORKLOADS[args.workload]()
        b, dt, frac, _ = oracle_throughput(wl, 10.0)
        line["cpu_baseline"] = {"value": round(b / dt / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"first {frac:.5f} of every matrix's rows + all activation "
                                          f"quantizations ({b} weight bytes in {dt:.1f} s, single thread)"}
        if not args.no_all_cores:
            try:
                b2, dt2, procs, frac2 = oracle_all_cores(wl, frac)
            except Exception as e:  # a worker that cannot start must not hold up the bench line
                b2 = None
                line["cpu_baseline"]["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
        if not args.no_all_cores and b2 is not None:
            line["cpu_baseline"]["all_cores"] = {
                "value": round(b2 / dt2 / 1e9, 6), "unit": "GB/s", "cores": procs, "host_cpus": os.cpu_count(),
                "sample": f"{procs} processes at once, each the first {frac2:.5f} of every matrix's rows + all "
                          f"activation quantizations ({b2} weight bytes, slowest process {dt2:.1f} s)"}
    if res.get("device_error"):
        line["device_error"] = res["device_error"]
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
