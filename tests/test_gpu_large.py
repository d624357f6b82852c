"""GPU parity for rank vectors larger than 4 GiB: 3 ranks of 2^30 + 37 int32
elements (4 GiB + 148 B each), so byte offsets pass 2^31 and 2^32 and every
32-bit index in a kernel would wrap.  Inputs follow a seeded closed-form
pattern written on the device; sampled outputs (uniform picks plus both sides
of the 2^31- and 2^32-byte marks, of every segment edge and of the vector's
end) are compared with the definition evaluated by the oracle on the same
sampled columns.  int32 sum and max are exact whatever the association
order, so every schedule and mode must match bit for bit.  Covers the fused
register path (AllReduce, ReduceScatter), the AllGather and the step
kernels (Ring AllReduce)."""
import numpy as np
import pytest

import hc_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

P = 3
N = (1 << 30) + 37
CHUNK = 1 << 26


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if torch.cuda.mem_get_info()[0] < 40 << 30:
        pytest.skip("needs 40 GiB of free device memory")
    from collective_communication_algorithms_gb300 import build
    build.build()


from collective_communication_algorithms_gb300 import _binding as B  # noqa: E402
from gpu_util import segments  # noqa: E402


def pattern_np(r, j):
    """Rank r's element j: a value in [-1000, 1000] (int64 arithmetic)."""
    j = np.asarray(j, dtype=np.int64)
    return ((j * 40503 + r * 7919 + (j >> 17) * 131) % 2001 - 1000).astype(np.int32)


def pattern_dev(r, out):
    """The same pattern written on the device, CHUNK elements at a time."""
    for s in range(0, out.numel(), CHUNK):
        j = torch.arange(s, min(s + CHUNK, out.numel()), dtype=torch.int64, device="cuda")
        out[s:s + j.numel()] = ((j * 40503 + r * 7919 + (j >> 17) * 131) % 2001 - 1000).to(torch.int32)


@pytest.fixture(scope="module")
def bufs():
    send = [torch.empty(N, dtype=torch.int32, device="cuda") for _ in range(P)]
    for r in range(P):
        pattern_dev(r, send[r])
    recv = [torch.empty(N, dtype=torch.int32, device="cuda") for _ in range(P)]
    torch.cuda.synchronize()
    yield send, recv
    del send, recv
    torch.cuda.empty_cache()


def sample(algo, coll):
    edges = [off for off, _ in segments(algo, coll, P, N, "int32")]
    edges += [1 << 29, 1 << 30, N]  # 2^31 and 2^32 bytes, the end
    J = hc_inputs.sample_indices(N, 4000, seed=7, segment_edges=edges)
    return J


def expected(J, op):
    Xs = np.stack([pattern_np(r, J) for r in range(P)])
    raw, _, _ = O.direct(Xs, op, "int32")
    return raw


def gather(t, J):
    return t[torch.from_numpy(J).cuda()].cpu().numpy()


@pytest.mark.parametrize("algo,mode", [("ring", "fused"), ("rhd", "fused"), ("ring", "step")])
@pytest.mark.parametrize("op", ["sum", "max"])
def test_allreduce_beyond_4GiB(bufs, algo, mode, op):
    send, recv = bufs
    for t in recv:
        t.fill_(0x5A5A5A5A)
    B.hc_allreduce([t.data_ptr() for t in send], [t.data_ptr() for t in recv], P, N, "int32", op,
                   algo, B.make_opts(mode), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    J = sample(algo, "allreduce")
    want = expected(J, op)
    for r in range(P):
        assert np.array_equal(gather(recv[r], J), want), (algo, mode, op, r)


def test_reducescatter_and_allgather_beyond_4GiB(bufs):
    send, recv = bufs
    segs = segments("ring", "reducescatter", P, N, "int32")
    out = [torch.full((max(ln, 4),), 0x5A5A5A5A, dtype=torch.int32, device="cuda") for _, ln in segs]
    B.hc_reduce_scatter([t.data_ptr() for t in send], [t.data_ptr() for t in out], P, N, "int32",
                        "sum", "ring", B.make_opts("fused"), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    J = sample("ring", "reducescatter")
    want = expected(J, "sum")
    for r, (off, ln) in enumerate(segs):
        m = (J >= off) & (J < off + ln)
        assert np.array_equal(gather(out[r], J[m] - off), want[m]), r
    # AllGather of the reduced segments (each segment is ~1.3 GiB)
    for t in recv:
        t.fill_(0x5A5A5A5A)
    B.hc_allgather([t.data_ptr() for t in out], [t.data_ptr() for t in recv], P, N, "int32", "ring",
                   B.make_opts("fused"), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    J = sample("ring", "allgather")
    want = expected(J, "sum")
    for r in range(P):
        assert np.array_equal(gather(recv[r], J), want), r
    assert B.hc_device_status() == 0
