"""hc_reduce_scatter_static_scratch: the ReduceScatter for callers that may
not allocate device memory (for example a plugin that its host framework
hands only input and output buffers, or a latency-critical path that cannot
afford cudaMalloc).  Its working memory is a fixed array inside the library,
so these tests check that it gives exactly what the ordinary entry point
gives with caller-provided scratch, on two calls in a row (the array keeps the
first call's contents), that it matches the oracle's replay directly, that a
call after the first on a device changes the device's free memory by not one
byte, and that work too large for the array is refused.

The file is named so that pytest collects it last.
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


def _rank_buffers(X):
    """(P, npad) device rows, 16-byte aligned, holding X."""
    P, n = X.shape
    npad = (n + 3) // 4 * 4
    t = torch.zeros((P, npad), dtype=torch.float32, device="cuda")
    t[:, :n] = torch.from_numpy(X).cuda()
    return t


def _outputs(algo, P, n):
    segs = [B.hc_segment_range(algo, "reducescatter", P, n, "float32", k) for k in range(P)]
    outs = [torch.full((max(ln, 4),), float("nan"), dtype=torch.float32, device="cuda")
            for _, ln in segs]
    return segs, outs


def _reduce_scatter_both_ways(algo, X, ranks_per_server=1, loop_bytes=0):
    P, n = X.shape
    src = _rank_buffers(X)
    sp = [src[r].data_ptr() for r in range(P)]
    stream = torch.cuda.current_stream().cuda_stream
    # existing entry point, step mode, caller-provided scratch
    segs, ref = _outputs(algo, P, n)
    need = B.hc_scratch_bytes(algo, P, n, "float32")
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    opts = B.make_opts("step", ranks_per_server=ranks_per_server, max_loop_bytes=loop_bytes,
                       scratch=scratch.data_ptr(), scratch_bytes=need)
    B.hc_reduce_scatter(sp, [t.data_ptr() for t in ref], P, n, "float32", "sum", algo, opts,
                        stream)
    # the allocation-free entry point
    _, got = _outputs(algo, P, n)
    B.hc_reduce_scatter_static_scratch(sp, [t.data_ptr() for t in got], P, n, "float32", "sum",
                                       algo, ranks_per_server, loop_bytes, stream)
    torch.cuda.synchronize()
    for r, (_, ln) in enumerate(segs):
        a = ref[r][:ln].cpu().numpy().view(np.uint32)
        b = got[r][:ln].cpu().numpy().view(np.uint32)
        assert np.array_equal(a, b), (algo, r)  # bit for bit, as every parity test here
    # the input is left untouched (out of place)
    assert np.array_equal(src[:, :n].cpu().numpy(), X)


def test_matches_existing_entry_point_on_two_calls_in_a_row():
    X1 = hc_inputs.gradients_f32(8, 300001, seed=21)
    X2 = hc_inputs.gradients_f32(8, 300001, seed=22)
    _reduce_scatter_both_ways("ring", X1)
    _reduce_scatter_both_ways("ring", X2)
    X3 = hc_inputs.gradients_f32(12, 100003, seed=23)
    _reduce_scatter_both_ways("rhd", X3)
    X4 = hc_inputs.gradients_f32(32, 50001, seed=24)
    _reduce_scatter_both_ways("pipeline", X4, ranks_per_server=8, loop_bytes=1 << 20)


def test_allocates_nothing_and_matches_the_oracle():
    """After a first call on the device (which, under lazy module loading,
    is where the array is committed), a second call leaves the device's free
    memory unchanged, and both calls' outputs equal the oracle's replay of
    the Ring ReduceScatter bit for bit."""
    P, n = 8, 300001
    X = hc_inputs.gradients_f32(P, n, seed=31)
    Y = O.replay("ring", "reducescatter", X, "sum", "float32")
    src = _rank_buffers(X)
    sp = [src[r].data_ptr() for r in range(P)]
    segs, outs = _outputs("ring", P, n)
    op = [t.data_ptr() for t in outs]
    stream = torch.cuda.current_stream().cuda_stream
    free = []
    for _ in range(2):
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        B.hc_reduce_scatter_static_scratch(sp, op, P, n, "float32", "sum", "ring", 1, 0, stream)
        torch.cuda.synchronize()
        for r, (off, ln) in enumerate(segs):
            got = outs[r][:ln].cpu().numpy().view(np.uint32)
            assert np.array_equal(got, Y[r, off:off + ln].view(np.uint32)), r
        for t in outs:
            t.fill_(float("nan"))
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
    assert free[1] == free[2], "the second call changed the device's free memory"


def test_rejects_work_larger_than_the_array():
    P = 8
    n = (32 << 20) // (4 * P) + 64  # 64 elements per rank more than the array holds
    assert B.hc_scratch_bytes("ring", P, n, "float32") > 32 << 20
    src = torch.zeros((P, n), dtype=torch.float32, device="cuda")
    segs, outs = _outputs("ring", P, n)
    with pytest.raises(B.HcError) as e:
        B.hc_reduce_scatter_static_scratch([src[r].data_ptr() for r in range(P)],
                                           [t.data_ptr() for t in outs], P, n, "float32", "sum",
                                           "ring")
    assert e.value.status == 4  # HC_ERR_SCRATCH
