"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times.  The oracle replays the schedule only on sampled element
indices (uniform picks plus both sides of every segment edge and of every
loop-slice edge); those outputs must match bit for bit.  The fp32/bf16
results are also checked over ALL elements against the fp64 direct sum:
normwise relative error <= 1e-5 (fp32) / 1e-2 (bf16) and, per element,
|y - y64| <= g_d * sum_i |x_i| with g_d = d u / (1 - d u) (d roundings on the
element's path).  Workloads:
  * int32 sum, values uniform in [-1000, 1000] from seed 0, 4096 elements:
    Ring over 4 ranks and RHD over 5 ranks, exact;
  * Ring AllReduce fp32 sum, P = 8, 16,777,216 elements per rank, N(0,1)*1e-3,
    plus ReduceScatter and AllGather alone on the same buffers;
  * RHD AllReduce fp32 sum, P in {5, 8, 12, 16}, 256 .. 16384 elements;
  * Ring and RHD AllReduce bf16, P = 8, 67,108,864 elements, N(0,1)*1e-2,
    sum and max;
  * Pipeline 4 x 8 (P = 32) fp32, 8,388,608 elements, N(0,1)*1e-3, AllReduce /
    ReduceScatter / AllGather, 64 MiB loop limit (4 loops with a tail).
"""
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
from gpu_util import run_collective, same_bits, segments  # noqa: E402


def sample(algo, coll, P, n, dtype, loop_bytes=0, p_intra=1, count=20000):
    segs = segments(algo, coll, P, n, dtype)
    edges = [off for off, _ in segs] + [off + ln for off, ln in segs]
    if loop_bytes:
        st, _ = B.hc_schedule_stats(algo, coll, P, n, dtype, p_intra, loop_bytes)
        for off, ln in segs:
            for i in range(1, st["loops"]):
                edges.append(off + i * st["chunk"])
    return hc_inputs.sample_indices(n, count, seed=P + n, segment_edges=edges)


def check_sampled(coll, algo, X, dtype, op, mode, p_intra=1, loop_bytes=0, in_place=False,
                  count=20000):
    P, n = X.shape
    res, ok = run_collective(coll, algo, X, dtype, op, mode, in_place, p_intra, loop_bytes)
    assert ok
    J = sample(algo, coll, P, n, dtype, loop_bytes, p_intra, count=count)
    Y = O.replay(algo, coll, X, op, dtype, p_intra=p_intra, loop_bytes=loop_bytes, J=J)
    segs = segments(algo, coll, P, n, dtype)
    for r in range(P):
        if coll == "reducescatter":
            off, ln = segs[r]
            m = (J >= off) & (J < off + ln)
            assert same_bits(res[r][J[m] - off], Y[r][m], dtype), (algo, coll, mode, r)
        else:
            assert same_bits(res[r][J], Y[r], dtype), (algo, coll, mode, r)
    return res


def depth(algo, P, p_intra):
    if algo == "ring":
        return P - 1
    if algo == "rhd":
        pp = 1 << (P.bit_length() - 1)
        return (pp.bit_length() - 1) + (1 if P > pp else 0)
    return (p_intra - 1) + (P // p_intra - 1)


def check_fp64(res0, X, dtype, algo, P, p_intra=1):
    _, y64, s1 = O.direct(X, "sum", dtype)
    if dtype == "float32":
        y = res0.view(np.float32).astype(np.float64)
        u, tol = 2.0 ** -24, 1e-5
    else:
        y = (res0.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        u, tol = 2.0 ** -8, 1e-2
    d = depth(algo, P, p_intra)
    g = d * u / (1 - d * u)
    assert np.linalg.norm(y - y64) / np.linalg.norm(y64) <= tol
    assert np.all(np.abs(y - y64) <= g * s1)


def test_int32_ring4_rhd5():
    X = hc_inputs.uniform_int32(5, 4096, seed=0)
    for mode in ("fused", "step"):
        res, ok = run_collective("allreduce", "ring", X[:4].copy(), "int32", "sum", mode)
        assert ok and all(np.array_equal(r.view(np.int32), X[:4].astype(np.int64).sum(0)) for r in res)
        res, ok = run_collective("allreduce", "rhd", X, "int32", "sum", mode)
        assert ok and all(np.array_equal(r.view(np.int32), X.astype(np.int64).sum(0)) for r in res)


@pytest.fixture(scope="module")
def ring_fp32_64MiB():
    return hc_inputs.gradients_f32(8, 16777216, seed=0, scale=1e-3)


@pytest.mark.parametrize("mode", ["fused", "step"])
def test_ring_fp32_64MiB(ring_fp32_64MiB, mode):
    X = ring_fp32_64MiB
    res = check_sampled("allreduce", "ring", X, "float32", "sum", mode)
    check_fp64(res[0], X, "float32", "ring", 8)
    check_sampled("reducescatter", "ring", X, "float32", "sum", mode)
    check_sampled("allgather", "ring", X, "float32", "sum", mode)


@pytest.mark.parametrize("P", [5, 8, 12, 16])
def test_rhd_small_messages(P):
    for n in (256, 512, 1024, 2048, 4096, 8192, 16384):
        X = hc_inputs.gradients_f32(P, n, seed=0, scale=1.0)
        Y = O.replay("rhd", "allreduce", X, "sum", "float32")
        for mode in ("fused", "step"):
            res, ok = run_collective("allreduce", "rhd", X, "float32", "sum", mode)
            assert ok and all(same_bits(res[r], Y[r], "float32") for r in range(P))
        st, _ = B.hc_schedule_stats("rhd", "allreduce", P, n, "float32")
        assert st["steps_per_loop"] == 2 * int(np.ceil(np.log2(P)))


@pytest.fixture(scope="module")
def bf16_128MiB():
    return hc_inputs.gradients_bf16(8, 67108864, seed=0, scale=1e-2)


@pytest.mark.parametrize("algo", ["ring", "rhd"])
@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("mode", ["fused", "step"])
def test_bf16_128MiB(bf16_128MiB, algo, op, mode):
    X = bf16_128MiB
    res = check_sampled("allreduce", algo, X, "bfloat16", op, mode, count=10000)
    if op == "sum":
        check_fp64(res[0], X, "bfloat16", algo, 8)
    else:
        raw, _, _ = O.direct(X[:, :1 << 20], "max", "bfloat16")
        assert np.array_equal(res[3][:1 << 20].view(np.uint16), raw)


@pytest.fixture(scope="module")
def pipe_fp32():
    return hc_inputs.gradients_f32(32, 8388608, seed=0, scale=1e-3)


@pytest.mark.parametrize("coll", ["allreduce", "reducescatter", "allgather"])
@pytest.mark.parametrize("mode", ["fused", "step"])
def test_pipeline_4x8(pipe_fp32, coll, mode):
    X = pipe_fp32
    lb = (64 << 20) if mode == "step" else 0
    st, _ = B.hc_schedule_stats("pipeline", coll, 32, 8388608, "float32", 8, 64 << 20)
    assert (st["loops"], st["tail"]) == (4, 37504)
    res = check_sampled(coll, "pipeline", X, "float32", "sum", mode, p_intra=8, loop_bytes=lb,
                        count=8000)
    if coll == "allreduce":
        check_fp64(res[0], X, "float32", "pipeline", 32, 8)
