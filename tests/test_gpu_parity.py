"""GPU parity: every algorithm x collective x dtype x op x mode, in place and
out of place, compared with the oracle's step-by-step replay element by
element, bit for bit, at sizes that span several tiles and a ragged tail;
plus the edge cases (empty input, P = 1, the maximum P = 64, one element).
All calls go through the C ABI (libhc.so)."""
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
    from collective_communication_algorithms_gb300 import _binding as B
    return B.lib()


from gpu_util import expected, run_collective, same_bits, segments  # noqa: E402

ALGOS = ("ring", "rhd", "pipeline")
COLLS = ("allreduce", "reducescatter", "allgather")
DTYPES = ("int32", "float32", "bfloat16")


def intra_for(algo, P):
    if algo != "pipeline":
        return 1
    for d in (8, 4, 3, 2):
        if P % d == 0 and P // d >= 2:
            return d
    return 1


def inputs(dtype, P, n, seed, op):
    if dtype == "int32":
        X = hc_inputs.uniform_int32(P, n, seed=seed)
        return (X % 5 + 1).astype(np.int32) if op == "prod" else X
    scale = 1.0
    X = hc_inputs.rank_buffers(dtype, P, n, seed=seed, scale=scale)
    if op == "prod" and dtype == "float32":
        X = (np.float32(1) + X * np.float32(0.01)).astype(np.float32)
    if op == "prod" and dtype == "bfloat16":
        X = hc_inputs.gradients_bf16(P, n, seed=seed, scale=0.01)
        X = (X.astype(np.uint32) | 0).astype(np.uint16)  # values near 0: product underflows gracefully
    return X


def check(coll, algo, X, dtype, op, mode, in_place, p_intra=1, loop_bytes=0):
    P, n = X.shape
    res, guards = run_collective(coll, algo, X, dtype, op, mode, in_place, p_intra, loop_bytes)
    assert guards, "a write landed outside its buffer"
    Y = O.replay(algo, coll, X, op, dtype, p_intra=p_intra, loop_bytes=loop_bytes)
    want = expected(coll, Y, segments(algo, coll, P, n, dtype) if coll != "allreduce" else None)
    for r in range(P):
        if not same_bits(res[r], want[r], dtype):
            a = res[r].view(np.int32 if dtype != "bfloat16" else np.int16)
            b = np.ascontiguousarray(want[r]).view(a.dtype)
            bad = np.nonzero(a != b)[0]
            raise AssertionError("%s %s %s %s %s P=%d n=%d rank %d: %d mismatches, first at %d"
                                 % (algo, coll, dtype, op, mode, P, n, r, bad.size, bad[0]))


SIZES = (1, 37, 4099, 65536 + 12)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_allreduce(algo, mode, dtype, op):
    for P in (2, 3, 5, 8, 12):
        pin = intra_for(algo, P)
        for n in SIZES:
            X = inputs(dtype, P, n, seed=P * 7 + n, op=op)
            for in_place in (False, True):
                check("allreduce", algo, X, dtype, op, mode, in_place, pin)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("coll", ["reducescatter", "allgather"])
def test_reducescatter_allgather(algo, mode, dtype, coll):
    for P in (2, 3, 5, 8, 12, 16):
        pin = intra_for(algo, P)
        for n in SIZES:
            X = inputs(dtype, P, n, seed=P * 11 + n, op="sum")
            for in_place in (False, True):
                check(coll, algo, X, dtype, "sum", mode, in_place, pin)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", COLLS)
def test_step_mode_loops(algo, coll):
    """Several loops with a tail slice; results equal the oracle's (which does
    not depend on the loops either)."""
    P = 8 if algo != "pipeline" else 8
    pin = intra_for(algo, P)
    n = 200003
    X = hc_inputs.gradients_f32(P, n, seed=3)
    for lb in (65536, 1 << 20):
        for in_place in (False, True):
            check(coll, algo, X, "float32", "sum", "step", in_place, pin, loop_bytes=lb)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("mode", ["fused", "step"])
def test_single_rank_and_max_ranks(algo, mode):
    for P in (1, 64):
        pin = intra_for(algo, P)
        for coll in COLLS:
            X = hc_inputs.gradients_f32(P, 3000, seed=P)
            for in_place in (False, True):
                check(coll, algo, X, "float32", "sum", mode, in_place, pin)


@pytest.mark.parametrize("algo", ALGOS)
def test_contribution_counting_int32(algo):
    """X_i = 2^i: every output is 2^P - 1 iff every rank contributed once."""
    for P in (2, 5, 8, 12, 16, 24, 30):
        pin = intra_for(algo, P)
        n = 4096 + 4
        X = np.tile((1 << np.arange(P, dtype=np.int64)).astype(np.int32)[:, None], (1, n))
        for mode in ("fused", "step"):
            res, ok = run_collective("allreduce", algo, X, "int32", "sum", mode, False, pin)
            assert ok
            for r in range(P):
                assert np.all(res[r].view(np.int32) == (1 << P) - 1), (algo, mode, P, r)


def test_empty_input_is_noop():
    from collective_communication_algorithms_gb300 import _binding as B
    B.hc_allreduce(None, None, 4, 0, "float32", "sum", "ring")
    B.hc_reduce_scatter(None, None, 4, 0, "float32", "sum", "rhd")
    B.hc_allgather(None, None, 4, 0, "float32", "pipeline")


def test_fused_and_step_agree_bitwise_tree_discriminating():
    """fp32 inputs mixing 2^24-scale values and small ones: any change of the
    association order shows up in low bits."""
    P, n = 12, 8192
    rng = np.random.default_rng(5)
    X = (rng.standard_normal((P, n)) * np.exp2(rng.integers(-20, 24, (P, n)))).astype(np.float32)
    for algo in ALGOS:
        pin = intra_for(algo, P)
        a, _ = run_collective("allreduce", algo, X, "float32", "sum", "fused", False, pin)
        b, _ = run_collective("allreduce", algo, X, "float32", "sum", "step", False, pin)
        for r in range(P):
            assert same_bits(a[r], b[r], "float32")
        check("allreduce", algo, X, "float32", "sum", "fused", False, pin)


def test_uses_the_given_stream():
    P, n = 4, 100000
    X = hc_inputs.gradients_f32(P, n, seed=1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        res, ok = run_collective("allreduce", "ring", X, "float32", "sum", "fused", False, 1,
                                 0, stream=s.cuda_stream)
    assert ok
    Y = O.replay("ring", "allreduce", X, "sum", "float32")
    assert same_bits(res[0], Y[0], "float32")


def _special_values(dtype, P, n, seed):
    """Bit patterns max/min must order by IEEE totalOrder: +-0, +-Inf, NaNs of
    both signs with several payloads, subnormals, the extremes, and random
    values, scattered over the ranks."""
    rng = np.random.default_rng(seed)
    if dtype == "bfloat16":
        pool = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F81, 0xFF81,
                         0x7FFF, 0xFFFF, 0x0001, 0x8001, 0x007F, 0x807F, 0x7F7F, 0xFF7F,
                         0x3F80, 0xBF80], dtype=np.uint16)
        X = rng.integers(0, 1 << 16, (P, n), dtype=np.uint32).astype(np.uint16)
    else:
        pool = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000,
                         0x7F800001, 0xFF800001, 0x7FFFFFFF, 0xFFFFFFFF, 0x00000001, 0x80000001,
                         0x007FFFFF, 0x807FFFFF, 0x7F7FFFFF, 0xFF7FFFFF, 0x3F800000, 0xBF800000],
                        dtype=np.uint32)
        X = rng.integers(0, 1 << 32, (P, n), dtype=np.uint64).astype(np.uint32)
    pick = rng.random((P, n)) < 0.5
    X[pick] = pool[rng.integers(0, pool.size, int(pick.sum()))]
    return X if dtype == "bfloat16" else X.view(np.float32)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("op", ["max", "min"])
def test_max_min_special_values(algo, dtype, op):
    """max / min of +-0, +-Inf, NaN payloads, subnormals and random bit
    patterns follow IEEE totalOrder bit for bit (oracle replay), fused and
    step mode, AllReduce and ReduceScatter."""
    for P in (3, 8, 12):
        pin = intra_for(algo, P)
        for n in (4099, 65548):
            X = _special_values(dtype, P, n, seed=P * 7 + n)
            for mode in ("fused", "step"):
                check("allreduce", algo, X, dtype, op, mode, False, pin)
                check("reducescatter", algo, X, dtype, op, mode, False, pin)


def test_concurrent_step_mode_calls_on_many_streams():
    """Small step-mode collectives (one programmatically dependent launch per
    step) issued on 6 streams at once, 40 calls each, every call on its own
    buffers: each result equals the oracle's and no device wait gave up."""
    from collective_communication_algorithms_gb300 import _binding as B
    P, n, calls = 8, 4099, 40
    streams = [torch.cuda.Stream() for _ in range(6)]
    jobs = []
    for i in range(len(streams) * calls):
        algo = ("ring", "rhd")[i % 2]
        X = hc_inputs.gradients_f32(P, n, seed=1000 + i)
        dev = [torch.from_numpy(X[r].copy()).cuda() for r in range(P)]  # one allocation per rank
        out = [torch.empty_like(d) for d in dev]
        jobs.append((algo, X, dev, out))
    torch.cuda.synchronize()
    opts = B.make_opts("step")
    for i, (algo, X, dev, out) in enumerate(jobs):
        s = streams[i % len(streams)]
        B.hc_allreduce([d.data_ptr() for d in dev], [o.data_ptr() for o in out],
                       P, n, "float32", "sum", algo, opts, s.cuda_stream)
    torch.cuda.synchronize()
    assert B.hc_device_status() == 0
    for algo, X, dev, out in jobs:
        Y = O.replay(algo, "allreduce", X, "sum", "float32")
        for r in range(P):
            assert same_bits(out[r].cpu().numpy(), Y[r], "float32"), (algo, r)


def test_concurrent_calls_from_host_threads():
    """Collectives issued from 6 host threads at once.  ctypes releases the
    interpreter lock during each call, so the library's host code (argument
    checks, step-plan cache, per-kernel attribute caches) runs concurrently.
    Each thread has its own stream and buffers and mixes schedules, modes and
    sizes, so plans are built and looked up concurrently; every result equals
    the oracle's."""
    import threading
    from collective_communication_algorithms_gb300 import _binding as B
    P, calls, nthreads = 8, 12, 6
    jobs = [[] for _ in range(nthreads)]
    for t in range(nthreads):
        for i in range(calls):
            j = t * calls + i
            algo = ("ring", "rhd", "pipeline")[j % 3]
            mode = ("fused", "step")[(j // 3) % 2]
            n = 4099 + 4 * (j % 5)  # a few sizes: plans shared and not shared between threads
            X = hc_inputs.gradients_f32(P, n, seed=5000 + j)
            dev = [torch.from_numpy(X[r].copy()).cuda() for r in range(P)]  # one allocation per rank
            out = [torch.empty_like(d) for d in dev]
            jobs[t].append((algo, mode, n, X, dev, out))
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(nthreads)

    def worker(t):
        try:
            s = torch.cuda.Stream()
            start.wait()
            for algo, mode, n, X, dev, out in jobs[t]:
                opts = B.make_opts(mode, ranks_per_server=2 if algo == "pipeline" else 1)
                B.hc_allreduce([d.data_ptr() for d in dev], [o.data_ptr() for o in out],
                               P, n, "float32", "sum", algo, opts, s.cuda_stream)
            s.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(nthreads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not errors, errors
    assert all(not th.is_alive() for th in threads)
    torch.cuda.synchronize()
    assert B.hc_device_status() == 0
    for t in range(nthreads):
        for algo, mode, n, X, dev, out in jobs[t]:
            Y = O.replay(algo, "allreduce", X, "sum", "float32", p_intra=2 if algo == "pipeline" else 1)
            for r in range(P):
                assert same_bits(out[r].cpu().numpy(), Y[r], "float32"), (t, algo, mode, n, r)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ("float32", "bfloat16"))
def test_fused_around_the_tma_rank_limit(algo, dtype):
    """Fused AllReduce and ReduceScatter with 17, 20, 32 and 33 ranks: the
    TMA-staged kernel up to 32 ranks (at 32 its P shared-memory tiles fill
    64 KB; RHD's 16-and-more-rank tree), the register path at 33.  Several
    tiles per segment and a ragged end; bit for bit against the oracle's
    replay, sum and max, in place and out of place."""
    for P in (17, 20, 32, 33):
        pin = intra_for(algo, P)
        n = P * 2048 + 13
        for op in ("sum", "max"):
            X = inputs(dtype, P, n, seed=P * 13 + 5, op=op)
            for in_place in (False, True):
                check("allreduce", algo, X, dtype, op, "fused", in_place, pin)
                check("reducescatter", algo, X, dtype, op, "fused", in_place, pin)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_tma_staged_paths(algo, dtype):
    """Segments of many 2 KB tiles of the TMA-staged fused reduce, with a
    partial last tile and a ragged end, for AllReduce and ReduceScatter
    (TMA-staged, and the register path where the library picks it: 4- and
    2-byte types, sum and max); the AllGather at twice the length (the
    register path at every rank count)."""
    from collective_communication_algorithms_gb300 import _binding as B
    per_seg = 70000 if dtype != "bfloat16" else 135000
    for P in (2, 3, 5, 8, 16, 17):
        pin = intra_for(algo, P) if algo != "pipeline" else (2 if P % 2 == 0 else 1)
        n = P * per_seg + 13
        for op in ("sum", "max"):
            X = inputs(dtype, P, n, seed=P + 101, op=op)
            for in_place in (False, True):
                check("allreduce", algo, X, dtype, op, "fused", in_place, pin)
                check("reducescatter", algo, X, dtype, op, "fused", in_place, pin)
        X = inputs(dtype, P, 2 * n, seed=P + 202, op="sum")
        for in_place in (False, True):
            check("allgather", algo, X, dtype, "sum", "fused", in_place, pin)
    assert B.hc_device_status() == 0


@pytest.mark.parametrize("algo", ("ring", "rhd"))
@pytest.mark.parametrize("dtype", DTYPES)
def test_large_narrow_step_launches(algo, dtype):
    """Step launches that move 8 MiB or more take the TMA-staged step kernel
    with 8 KB tiles even when their items are narrow (one input and an
    accumulator, or a copy): segments ending in a partial tile, a ragged end
    of the rank vector, RHD's fold and unfold (P = 5), in-place AllReduce,
    sum and max."""
    from collective_communication_algorithms_gb300 import _binding as B
    per_seg = 350003 if dtype != "bfloat16" else 700001
    for P in (5, 8):
        n = P * per_seg + 13
        for op in ("sum", "max"):
            X = inputs(dtype, P, n, seed=P + 303, op=op)
            for in_place in (False, True):
                check("allreduce", algo, X, dtype, op, "step", in_place)
        X = inputs(dtype, P, n, seed=P + 404, op="sum")
        check("reducescatter", algo, X, dtype, "sum", "step", False)
        check("allgather", algo, X, dtype, "sum", "step", False)
    assert B.hc_device_status() == 0


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_broadcast(mode, dtype):
    """RHD Broadcast: every rank ends with the root's vector, bit for bit."""
    for P in (1, 2, 3, 5, 8, 12, 16):
        roots = range(P) if P <= 8 else (0, 1, P // 2, P - 1)
        # 300,007 elements: many blocks per segment
        for n in (1, 37, 4099, 80000 + 3, 300007):
            X = inputs(dtype, P, n, seed=P * 13 + n, op="sum")
            for root in roots:
                for in_place in (False, True):
                    res, ok = run_collective("broadcast", "rhd", X, dtype, mode=mode,
                                             in_place=in_place, root=root)
                    assert ok, "a write landed outside its buffer"
                    Y = O.replay("rhd", "broadcast", X, "sum", dtype, root=root)
                    for r in range(P):
                        assert same_bits(res[r], Y[r], dtype), (P, n, root, r, in_place)


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_hierarchical_allreduce(mode, dtype, op):
    """Plain hierarchical AllReduce (mesh RS, inter-server RHD AR, mesh AG)
    against the oracle, bit for bit."""
    for P, pin in ((4, 4), (6, 3), (8, 2), (8, 4), (12, 4), (20, 4), (32, 8), (64, 8)):
        for n in (37, 4099, 65536 + 12):
            X = inputs(dtype, P, n, seed=P * 17 + n, op=op)
            for in_place in (False, True):
                check("allreduce", "hier", X, dtype, op, mode, in_place, pin)
    X = inputs(dtype, 12, 200003, seed=5, op=op)
    check("allreduce", "hier", X, dtype, op, "step", False, 4, loop_bytes=1 << 20)


def test_zz_no_device_timeouts_recorded():
    """No bounded device-side wait gave up during the GPU tests above."""
    from collective_communication_algorithms_gb300 import _binding as B
    assert B.hc_device_status(clear=False) == 0


def test_bound_calls_equal_plain_calls():
    """BoundCall objects (arguments converted once, the call repeated) give
    bit for bit what the plain entry points give, call after call."""
    from collective_communication_algorithms_gb300 import _binding as B
    P, n = 8, 40000
    X = hc_inputs.gradients_f32(P, n, seed=77)
    dev = torch.from_numpy(X).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for algo, mode in (("ring", "fused"), ("rhd", "step"), ("pipeline", "step")):
        opts = B.make_opts(mode, ranks_per_server=4 if algo == "pipeline" else 1)
        a, b = torch.zeros_like(dev), torch.zeros_like(dev)
        rows = lambda t: [t[r].data_ptr() for r in range(P)]
        B.hc_allreduce(rows(dev), rows(a), P, n, "float32", "sum", algo, opts, stream)
        call = B.bind_allreduce(rows(dev), rows(b), P, n, "float32", "sum", algo, opts, stream)
        for _ in range(3):
            b.zero_()
            call()
            torch.cuda.synchronize()
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), (algo, mode)
    assert B.hc_device_status() == 0

