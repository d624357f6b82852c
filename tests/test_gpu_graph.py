"""Graph mode on the GPU: a DAG of collectives (fused and step mode,
dependent and independent) built once and launched twice gives, bit for bit,
what the same collectives give run eagerly in the order added, and the
oracle's result."""
import numpy as np
import pytest

import hc_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from collective_communication_algorithms_gb300 import build
    build.build()


from collective_communication_algorithms_gb300 import _binding as B  # noqa: E402


def rows(t):
    return [t[r].data_ptr() for r in range(t.shape[0])]


def run_sequence(use_graph, X, launches=1):
    """AR(X->Y, ring fused); AR(Z in place, rhd step); RS(Y->W, ring fused);
    AG(W in place, pipeline 2 x 4, step); AR(Z->V, max, pipeline 2 x 4, fused)."""
    P, n = X.shape
    dev = torch.from_numpy(X).cuda()
    Y = torch.zeros_like(dev)
    Z = dev.clone()
    V = torch.zeros_like(dev)
    W = torch.zeros_like(dev)
    segs = [B.hc_segment_range("ring", "reducescatter", P, n, "float32", k) for k in range(P)]
    w_seg = [W[r].data_ptr() + segs[r][0] * 4 for r in range(P)]
    step = B.make_opts("step")
    pipe_step = B.make_opts("step", ranks_per_server=4)
    pipe_fused = B.make_opts("fused", ranks_per_server=4)
    calls = [
        ("ar", rows(dev), rows(Y), "sum", "ring", None),
        ("ar", rows(Z), rows(Z), "sum", "rhd", step),
        ("rs", rows(Y), w_seg, "sum", "ring", None),
        ("ag", w_seg, rows(W), None, "pipeline", pipe_step),
        ("ar", rows(Z), rows(V), "max", "pipeline", pipe_fused),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    if use_graph:
        g = B.Graph()
        for kind, s, r, op, algo, opts in calls:
            if kind == "ar":
                g.add_allreduce(s, r, P, n, "float32", op, algo, opts)
            elif kind == "rs":
                g.add_reduce_scatter(s, r, P, n, "float32", op, algo, opts)
            else:
                g.add_allgather(s, r, P, n, "float32", algo, opts)
        g.build()
        info = g.info()
        for _ in range(launches):
            g.launch(stream)
        torch.cuda.synchronize()
        g.close()
    else:
        info = None
        for kind, s, r, op, algo, opts in calls:
            if kind == "ar":
                B.hc_allreduce(s, r, P, n, "float32", op, algo, opts, stream)
            elif kind == "rs":
                B.hc_reduce_scatter(s, r, P, n, "float32", op, algo, opts, stream)
            else:
                B.hc_allgather(s, r, P, n, "float32", algo, opts, stream)
        torch.cuda.synchronize()
    out = {k: t.cpu().numpy() for k, t in (("Y", Y), ("Z", Z), ("V", V), ("W", W))}
    return out, info


def test_graph_equals_eager_and_oracle():
    P, n = 8, 100000
    X = hc_inputs.gradients_f32(P, n, seed=31)
    eager, _ = run_sequence(False, X)
    graph, info = run_sequence(True, X)
    assert info["collectives"] == 5
    assert info["edges"] >= 3 and info["kernels"] >= 5
    for k in eager:
        assert np.array_equal(eager[k].view(np.uint32), graph[k].view(np.uint32)), k
    Y = O.replay("ring", "allreduce", X, "sum", "float32")
    assert np.array_equal(graph["Y"].view(np.uint32), Y.view(np.uint32))
    Z = O.replay("rhd", "allreduce", X, "sum", "float32")
    assert np.array_equal(graph["Z"].view(np.uint32), Z.view(np.uint32))
    V = O.replay("pipeline", "allreduce", Z, "max", "float32", p_intra=4)
    assert np.array_equal(graph["V"].view(np.uint32), V.view(np.uint32))
    assert B.hc_device_status() == 0


def test_graph_replays():
    """Launching an in-place AllReduce graph twice applies it twice."""
    P, n = 4, 4096
    X = hc_inputs.uniform_int32(P, n, seed=3)
    dev = torch.from_numpy(X).cuda()
    g = B.Graph()
    g.add_allreduce(rows(dev), rows(dev), P, n, "int32", "sum", "ring", B.make_opts("step"))
    g.add_allreduce(rows(dev), rows(dev), P, 0, "int32", "sum", "ring")  # empty: no kernels
    g.build()
    stream = torch.cuda.current_stream().cuda_stream
    g.launch(stream)
    g.launch(stream)
    torch.cuda.synchronize()
    got = dev.cpu().numpy()
    want = (X.astype(np.int64).sum(0) * P).astype(np.int32)
    assert all(np.array_equal(got[r], want) for r in range(P))
    g.close()


@pytest.mark.parametrize("use_graph", [False, True])
def test_chained_step_calls_read_the_previous_calls_output(use_graph):
    """Step-mode calls load the inputs no launch of the call writes before
    waiting for the previous launch (from a call's second launch on).  Two
    Pipeline 2 x 4 AllReduces (TMA-staged mesh reduce steps) and a
    hierarchical one, each reading the previous call's output, queued on one
    stream with no synchronisation in between (eagerly, or as one graph):
    every result equals the oracle's replay of the chain, bit for bit."""
    P, n = 8, 70000 + 3
    npad = (n + 3) // 4 * 4  # rows start on 16-byte boundaries; the calls use n
    X = hc_inputs.gradients_f32(P, n, seed=41)
    dev = torch.zeros((P, npad), dtype=torch.float32, device="cuda")
    dev[:, :n] = torch.from_numpy(X).cuda()
    A, Bv, C = torch.zeros_like(dev), torch.zeros_like(dev), torch.zeros_like(dev)
    pipe = B.make_opts("step", ranks_per_server=4, max_loop_bytes=256 << 10)
    hier = B.make_opts("step", ranks_per_server=4)
    calls = [(rows(dev), rows(A), "pipeline", pipe), (rows(A), rows(Bv), "pipeline", pipe),
             (rows(Bv), rows(C), "hier", hier)]
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    if use_graph:
        g = B.Graph()
        for s, r, algo, opts in calls:
            g.add_allreduce(s, r, P, n, "float32", "sum", algo, opts)
        g.build()
        assert g.info()["edges"] >= 2
        g.launch(stream)
        torch.cuda.synchronize()
        g.close()
    else:
        for s, r, algo, opts in calls:
            B.hc_allreduce(s, r, P, n, "float32", "sum", algo, opts, stream)
        torch.cuda.synchronize()
    Y1 = O.replay("pipeline", "allreduce", X, "sum", "float32", p_intra=4, loop_bytes=256 << 10)
    Y2 = O.replay("pipeline", "allreduce", Y1, "sum", "float32", p_intra=4, loop_bytes=256 << 10)
    Y3 = O.replay("hier", "allreduce", Y2, "sum", "float32", p_intra=4)
    for got, want in ((A, Y1), (Bv, Y2), (C, Y3)):
        assert np.array_equal(got[:, :n].cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert B.hc_device_status() == 0


@pytest.mark.parametrize("use_graph", [False, True])
def test_chained_large_narrow_step_calls(use_graph):
    """The same for Ring and RHD step calls whose launches move 8 MiB or
    more and so run on the TMA-staged step kernel with 8 KB tiles, loading
    the call's own inputs early: Ring, RHD and Ring AllReduces chained on
    one stream (eagerly, or as one graph), each reading the previous call's
    output; every result equals the oracle's replay of the chain."""
    P, n = 8, 8 * 350003 + 13
    npad = (n + 3) // 4 * 4
    X = hc_inputs.gradients_f32(P, n, seed=43)
    dev = torch.zeros((P, npad), dtype=torch.float32, device="cuda")
    dev[:, :n] = torch.from_numpy(X).cuda()
    A, Bv, C = torch.zeros_like(dev), torch.zeros_like(dev), torch.zeros_like(dev)
    step = B.make_opts("step")
    calls = [(rows(dev), rows(A), "ring"), (rows(A), rows(Bv), "rhd"), (rows(Bv), rows(C), "ring")]
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    if use_graph:
        g = B.Graph()
        for s_, r_, algo in calls:
            g.add_allreduce(s_, r_, P, n, "float32", "sum", algo, step)
        g.build()
        assert g.info()["edges"] >= 2
        g.launch(stream)
        torch.cuda.synchronize()
        g.close()
    else:
        for s_, r_, algo in calls:
            B.hc_allreduce(s_, r_, P, n, "float32", "sum", algo, step, stream)
        torch.cuda.synchronize()
    Y1 = O.replay("ring", "allreduce", X, "sum", "float32")
    Y2 = O.replay("rhd", "allreduce", Y1, "sum", "float32")
    Y3 = O.replay("ring", "allreduce", Y2, "sum", "float32")
    for got, want in ((A, Y1), (Bv, Y2), (C, Y3)):
        assert np.array_equal(got[:, :n].cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert B.hc_device_status() == 0
