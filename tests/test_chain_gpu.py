"""Chained decode steps (qgemv_chain_*) on the GPU.

Every output of a chain must equal, bit for bit, what the corresponding single calls issued in order on one
stream produce (a chain step runs the same staging, decode and per-row arithmetic), and a step must see
the outputs of every earlier step (the grid-wide barrier between steps).
"""
import numpy as np
import pytest

import oracle
import qgemv_inputs as gen
import quantized_weight_gemv_quantize_gb300 as qg

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qg.build()
    qg.lib()
    qg.qgemv_device_error(reset=True)
    yield
    assert qg.qgemv_device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def table_for(n):
    return torch.zeros(qg.qgemv_chain_bytes(n), dtype=torch.uint8, device="cuda")


def f32(K, seed):
    return dev(gen.normal_f32(K, seed))


def test_chain_equals_single_calls_for_mixed_steps():
    # quantize (K=3072) -> Q6_K on it; Q4_K over three matrices with fp32 input quantized in the launch and
    # published; Q8_0 on the published blocks; Q5_K with fp32 input; Q4_K on a long row (multi-warp teams)
    x0, x1, x2, x3 = f32(3072, 1), f32(1024, 2), f32(2560, 3), f32(4096, 4)
    W6 = dev(gen.weights("Q6_K", 1024, 3072, 11))
    W4 = [dev(gen.weights("Q4_K", N, 1024, 12 + j)) for j, N in enumerate((2048, 1024, 1024))]
    W8 = dev(gen.weights("Q8_0", 5000, 1024, 13))
    W5 = dev(gen.weights("Q5_K", 777, 2560, 14))
    W4b = dev(gen.weights("Q4_K", 333, 4096, 15))

    def outs():
        return dict(y6=torch.full((1024,), float("nan"), device="cuda"),
                    y4=[torch.full((N,), float("nan"), device="cuda") for N in (2048, 1024, 1024)],
                    y8=torch.full((5000,), float("nan"), device="cuda"),
                    y5=torch.full((777,), float("nan"), device="cuda"),
                    y4b=torch.full((333,), float("nan"), device="cuda"),
                    xq0=torch.zeros(qg.qgemv_act_bytes(1, 3072), dtype=torch.uint8, device="cuda"),
                    xq1=torch.zeros(qg.qgemv_act_bytes(1, 1024), dtype=torch.uint8, device="cuda"))

    ref = outs()
    qg.qgemv_quantize_act(x0, 1, 3072, ref["xq0"])
    qg.qgemv("Q6_K", W6, ref["xq0"], ref["y6"], 1, 1024, 3072)
    qg.qgemv_multi("Q4_K", [(W, y, N) for W, y, N in zip(W4, ref["y4"], (2048, 1024, 1024))], "f32", x1, 1, 1024,
                   xq_out=ref["xq1"])
    qg.qgemv("Q8_0", W8, ref["xq1"], ref["y8"], 1, 5000, 1024)
    qg.qgemv_multi("Q5_K", [(W5, ref["y5"], 777)], "f32", x2, 1, 2560)
    qg.qgemv_multi("Q4_K", [(W4b, ref["y4b"], 333)], "f32", x3, 1, 4096)
    torch.cuda.synchronize()

    got = outs()
    steps = [("quantize", x0, 3072, got["xq0"]),
             ("gemv", "Q6_K", "q8_1", got["xq0"], 3072, [(W6, got["y6"], 1024)], None),
             ("gemv", "Q4_K", "f32", x1, 1024, [(W, y, N) for W, y, N in zip(W4, got["y4"], (2048, 1024, 1024))],
              got["xq1"]),
             ("gemv", "Q8_0", "q8_1", got["xq1"], 1024, [(W8, got["y8"], 5000)], None),
             ("gemv", "Q5_K", "f32", x2, 2560, [(W5, got["y5"], 777)], None),
             ("gemv", "Q4_K", "f32", x3, 4096, [(W4b, got["y4b"], 333)], None)]
    table = table_for(len(steps))
    qg.qgemv_chain_prepare(steps, table)
    for run in range(3):  # the barrier state carries over from run to run
        for v in (got["y6"], got["y8"], got["y5"], got["y4b"], *got["y4"]):
            v.fill_(float("nan"))
        qg.qgemv_route_reset()
        qg.qgemv_chain_run(table)
        torch.cuda.synchronize()
        assert qg.qgemv_route_counts()[qg.ROUTE_CHAIN] == 1
        assert torch.equal(got["xq0"], ref["xq0"]) and torch.equal(got["xq1"], ref["xq1"])
        for k in ("y6", "y8", "y5", "y4b"):
            assert torch.equal(got[k], ref[k]), (run, k)
        for a, b in zip(got["y4"], ref["y4"]):
            assert torch.equal(a, b), run
    qg.qgemv_chain_release(table)
    with pytest.raises(qg.QgemvError):
        qg.qgemv_chain_run(table)


def test_chain_step_reads_the_previous_steps_output():
    # y_i = W_i xhat(y_{i-1}): every GEMV reads the fp32 output of the step before it, so a step that ran
    # ahead of the barrier would read a stale or partly written input
    n, K = 24, 1024
    Ws = [dev(gen.weights("Q8_0", K, K, 300 + i)) for i in range(n)]
    x = f32(K, 299)
    ref = [torch.empty(K, device="cuda") for _ in range(n)]
    prev = x
    for i in range(n):
        qg.qgemv_multi("Q8_0", [(Ws[i], ref[i], K)], "f32", prev, 1, K)
        prev = ref[i]
    torch.cuda.synchronize()
    ys = [torch.full((K,), float("nan"), device="cuda") for _ in range(n)]
    steps = []
    prev = x
    for i in range(n):
        steps.append(("gemv", "Q8_0", "f32", prev, K, [(Ws[i], ys[i], K)], None))
        prev = ys[i]
    table = table_for(n)
    qg.qgemv_chain_prepare(steps, table)
    for _ in range(5):
        for y in ys:
            y.fill_(float("nan"))
        qg.qgemv_chain_run(table)
        torch.cuda.synchronize()
        for i in range(n):
            assert torch.equal(ys[i], ref[i]), i
    assert np.isfinite(ys[-1].cpu().numpy()).all()
    qg.qgemv_chain_release(table)


def test_chain_matches_the_oracle():
    K, N = 2560, 4096
    W = gen.weights("Q4_K", N, K, 77)
    xh = gen.normal_f32(K, 78)
    y = torch.full((N,), float("nan"), device="cuda")
    xq = torch.zeros(qg.qgemv_act_bytes(1, K), dtype=torch.uint8, device="cuda")
    steps = [("quantize", dev(xh), K, xq), ("gemv", "Q4_K", "q8_1", xq, K, [(dev(W), y, N)], None)]
    table = table_for(2)
    qg.qgemv_chain_prepare(steps, table)
    qg.qgemv_chain_run(table)
    torch.cuda.synchronize()
    xq_ref = oracle.quantize_act(xh.reshape(1, K))
    assert np.array_equal(xq.cpu().numpy(), xq_ref.reshape(-1))
    ref = oracle.gemv("Q4_K", W, xq_ref, 1, N, K)[0]
    err = y.cpu().numpy().astype(np.float64) - ref
    assert np.linalg.norm(err) <= 1e-5 * np.linalg.norm(ref)
    assert np.abs(err).max() <= 1e-3 * np.linalg.norm(ref)
    qg.qgemv_chain_release(table)


def test_chain_replays_in_a_cuda_graph():
    K = 1024
    Ws = [dev(gen.weights("Q4_K", 2048, K, 400 + i)) for i in range(4)]
    x = f32(K, 401)
    ys = [torch.full((2048,), float("nan"), device="cuda") for _ in range(4)]
    steps = [("gemv", "Q4_K", "f32", x, K, [(W, y, 2048)], None) for W, y in zip(Ws, ys)]
    table = table_for(4)
    qg.qgemv_chain_prepare(steps, table)
    qg.qgemv_chain_run(table)
    torch.cuda.synchronize()
    ref = [y.clone() for y in ys]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            qg.qgemv_chain_run(table, stream=s)
            qg.qgemv_chain_run(table, stream=s)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for y, r in zip(ys, ref):
            assert torch.equal(y, r)
    qg.qgemv_chain_release(table)
