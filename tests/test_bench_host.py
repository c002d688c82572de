"""Host-side logic of the benchmark's multi-process path, run as world-size-2 gloo ranks on CPU.

Every rank sweeps the full weight set (replicas; no collective on the data path); the step time is the
slowest rank's, and rank 0 reports N x weight bytes / that time.  The oracle's reference arm runs on
rank 0 only.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [0.75, 1.25][rank]  # ms per step seen by this rank
        ms = bench.max_over_ranks(local, dist, "cpu")
        dist.barrier()
        args = bench.argparse.Namespace(gpus=world, steps=3, warmup=3, workload="dense-q4k-256x1024")
        ref = bench.run_reference(args, rank, world) if rank != 0 else "skipped-on-rank-0"
        out.put((rank, ms, bench.sweep_value(world, 10**9, ms), ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_report_the_whole_job():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [1.25, 1.25]                 # both ranks see the max
    assert res[0][2] == pytest.approx(2 * 1.0 / 1.25e-3)       # 2 replicas x 1 GB per 1.25 ms, in GB/s
    assert res[1][3] is None                                   # reference arm: rank 1 does no work


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.sweep_value(1, 435740672, 0.5) == pytest.approx(871.481344)


def test_traffic_rows_apply_only_to_their_build(tmp_path, monkeypatch):
    # a row of the traffic table is used only for its workload, kernel class and source hash
    h = bench.kernel_source_hash()
    (tmp_path / "traffic.md").write_text(
        "| workload | kernel | bytes per launch | source hash |\n|---|---|---|---|\n"
        f"| wl-a | Q4_K/m1 | 1234 | {h} |\n| wl-a | Q6_K/m1 | 99 | 000000000000 |\n")
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.traffic_from_profiles("wl-a", "Q4_K/m1") == 1234.0
    assert bench.traffic_from_profiles("wl-a", "Q6_K/m1") is None     # captured from another build
    assert bench.traffic_from_profiles("wl-b", "Q4_K/m1") is None     # another workload


def test_source_hash_ignores_comments_and_trace_blocks_but_not_code(tmp_path, monkeypatch):
    import shutil
    root = tmp_path / "r"
    shutil.copytree(os.path.join(bench.ROOT, "quantized_weight_gemv_quantize_gb300", "csrc"),
                    root / "quantized_weight_gemv_quantize_gb300" / "csrc")
    (root / "include").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "include", "qgemv.h"), root / "include" / "qgemv.h")
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    f = root / "quantized_weight_gemv_quantize_gb300" / "csrc" / "common.cuh"
    f.write_text(f.read_text() + "\n// a remark\n/* another */\n")
    assert bench.kernel_source_hash() == h0
    f.write_text(f.read_text() + "\n#ifdef QGEMV_TRACE\nconstexpr int kTraceOnly = 1;\n#endif\n")
    assert bench.kernel_source_hash() == h0                       # timeline-build code is not compiled
    f.write_text(f.read_text() + "\n#ifdef QGEMV_TRACE\nint a;\n#else\nint b;\n#endif\n")
    assert bench.kernel_source_hash() != h0                       # its #else part is
    f.write_text(f.read_text() + "\nconstexpr int kChanged = 1;\n")
    assert bench.kernel_source_hash() != h0


def test_kernel_launch_count_excludes_attribute_counters():
    import quantized_weight_gemv_quantize_gb300 as qg

    class FakeLib:
        ROUTE_FUSED, ROUTE_GROUPED, ROUTE_PDL, ROUTE_ARGMAX, ROUTE_CHUNKED = (
            qg.ROUTE_FUSED, qg.ROUTE_GROUPED, qg.ROUTE_PDL, qg.ROUTE_ARGMAX, qg.ROUTE_CHUNKED)

        def __init__(self):
            self.c = [0] * qg.NUM_ROUTES

        def qgemv_route_reset(self):
            self.c = [0] * qg.NUM_ROUTES

        def qgemv_route_counts(self):
            return list(self.c)

    class FakeStream:
        def synchronize(self):
            pass

    lib = FakeLib()

    def run():  # a quantize launch, a Q4_K m=1 GEMV with PDL, and a 16-row call served as two launches
        lib.c[0] += 1
        lib.c[1] += 1
        lib.c[qg.ROUTE_PDL] += 2
        lib.c[8] += 1
        lib.c[8] += 1
        lib.c[qg.ROUTE_FUSED] += 1

    assert bench.kernel_launches(lib, run, FakeStream()) == 4


def test_reference_arm_prints_one_contract_line():
    # the reference arm (the CPU oracle) runs without a GPU: one JSON line with the contract's keys
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload",
                        "dense-q4k-256x1024", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["gpu_launches"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "dense-q4k-256x1024"


class _FakeBuffer:
    """Stand-in for a device buffer: building the call list only reads its address."""

    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def _host_sweep(name):
    import quantized_weight_gemv_quantize_gb300 as qg
    from qgemv_inputs.workloads import WORKLOADS
    sw = object.__new__(bench.Sweep)
    sw.wl, sw.qg, sw.L, sw.fuse_max = WORKLOADS[name](), qg, qg.lib(), bench.Sweep.FUSE_MAX_DEFAULT
    sw._layout(sw.wl, qg)
    sw.wbuf, sw.d_in, sw.d_xq, sw.d_out = (_FakeBuffer(a << 32) for a in (1, 2, 3, 4))
    return sw


@pytest.mark.parametrize("mode", ["fused", "percall"])
def test_sweep_gives_the_late_trigger_only_to_quantize_launches_before_short_gemvs(mode):
    import quantized_weight_gemv_quantize_gb300 as qg
    pdl, late = qg.QGEMV_FLAG_PDL, qg.QGEMV_FLAG_PDL_LATE_TRIGGER
    for name in ("dense-0.6b-class", "dense-4b-class"):
        sw = _host_sweep(name)
        calls = sw.calls(mode, True)
        quant = [j for j, c in enumerate(calls) if c[0] == "quantize"]
        assert quant
        for j in quant:
            flags = sw.calls(mode, False)[j][2][4]
            assert flags == 0  # without PDL no launch flag at all
            flags = calls[j][2][4]
            # the launch that reads the quantized activation is the next one; its weights decide (its
            # algorithmic bytes: the weights plus a few KB of activation and outputs, and no launch of these
            # sweeps is within a few KB of the threshold)
            nxt = calls[j + 1]
            wbytes = nxt[3]
            short = wbytes < bench.SHORT_GEMV_BYTES
            assert flags == (pdl | late if short else pdl), (name, mode, j, nxt[0], wbytes)
        if name == "dense-4b-class":
            assert all(calls[j][2][4] == pdl for j in quant)  # every 4B-class GEMV streams 6-319 MB
        elif mode == "fused":
            assert all(calls[j][2][4] == pdl | late for j in quant)  # each precedes a 2.6 MB down projection
