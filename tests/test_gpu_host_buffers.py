"""Page-locked host buffers (hc_opts_t.host_buffers = 1): the kernels read and
write pinned host memory directly over the host link.  Results are compared
with the oracle's replay bit for bit, every buffer carries guard bands, and
pageable memory is refused before anything is launched."""
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


from gpu_util import CANARY, ESIZE, GUARD, NP_INT, TORCH_INT, expected, same_bits, segments  # noqa: E402


class HostRegion:
    """A pinned host buffer of `length` elements with guard bands on both
    sides, 16-byte aligned at its first element."""

    def __init__(self, dtype, length):
        A = 16 // ESIZE[dtype]
        self.dtype = dtype
        self.length = length
        self.t = torch.empty(GUARD + ((length + A - 1) // A) * A + GUARD,
                             dtype=TORCH_INT[dtype]).pin_memory()
        self.t.fill_(np.array(CANARY[dtype]).astype(NP_INT[dtype]).item())
        self.ptr = self.t.data_ptr() + GUARD * ESIZE[dtype]
        assert self.ptr % 16 == 0

    def write(self, arr):
        a = np.ascontiguousarray(arr).view(NP_INT[self.dtype])
        self.t[GUARD:GUARD + a.size] = torch.from_numpy(a.copy())

    def read(self, at=0, length=None):
        length = self.length - at if length is None else length
        return self.t[GUARD + at:GUARD + at + length].numpy().copy()

    def guards_ok(self):
        h = self.t.numpy()
        c = np.array(CANARY[self.dtype]).astype(NP_INT[self.dtype])
        return bool(np.all(h[:GUARD] == c) and np.all(h[GUARD + self.length:] == c))


def run_host(coll, algo, X, dtype, op, mode, p_intra=1, root=0, recv_on_device=False):
    """One collective with its inputs (and outputs, unless recv_on_device) in
    pinned host memory.  Returns (per-rank results, guards ok)."""
    from collective_communication_algorithms_gb300 import _binding as B
    from gpu_util import Region
    P, n = X.shape
    segs = segments(algo, coll, P, n, dtype) if coll in ("reducescatter", "allgather") else None
    regions = []
    if coll == "allgather":
        send = []
        for k in range(P):
            off, ln = segs[k]
            s = HostRegion(dtype, ln)
            s.write(X[k, off:off + ln])
            regions.append(s)
            send.append(s.ptr)
    elif coll == "broadcast":
        s = HostRegion(dtype, n)
        s.write(X[root])
        regions.append(s)
        send = s.ptr
    else:
        send = []
        for r in range(P):
            s = HostRegion(dtype, n)
            s.write(X[r])
            regions.append(s)
            send.append(s.ptr)
    out_len = [segs[r][1] if coll == "reducescatter" else n for r in range(P)]
    mk = (lambda ln: Region(dtype, ln)) if recv_on_device else (lambda ln: HostRegion(dtype, ln))
    outs = [mk(out_len[r]) for r in range(P)]
    regions += outs
    recv = [o.ptr for o in outs]
    scratch = None
    sp, sb = 0, 0
    if coll == "reducescatter" and mode == "step":
        sb = B.hc_scratch_bytes(algo, P, n, dtype)
        scratch = torch.empty(max(sb, 16), dtype=torch.uint8, device="cuda")
        sp = scratch.data_ptr()
    opts = B.make_opts(mode, ranks_per_server=p_intra, scratch=sp, scratch_bytes=sb,
                       host_buffers=True)
    torch.cuda.synchronize()
    if coll == "allreduce":
        B.hc_allreduce(send, recv, P, n, dtype, op, algo, opts, 0)
    elif coll == "reducescatter":
        B.hc_reduce_scatter(send, recv, P, n, dtype, op, algo, opts, 0)
    elif coll == "allgather":
        B.hc_allgather(send, recv, P, n, dtype, algo, opts, 0)
    else:
        B.hc_broadcast(send, recv, P, n, dtype, root, algo, opts, 0)
    torch.cuda.synchronize()
    res = [o.read(0, out_len[r]) for r, o in enumerate(outs)]
    return res, all(g.guards_ok() for g in regions)


def check_host(coll, algo, X, dtype, op, mode, p_intra=1, root=0, recv_on_device=False):
    P, n = X.shape
    res, ok = run_host(coll, algo, X, dtype, op, mode, p_intra, root, recv_on_device)
    assert ok, "a write landed outside its buffer"
    Y = O.replay(algo, coll, X, op, dtype, p_intra=p_intra, root=root)
    want = expected(coll, Y, segments(algo, coll, P, n, dtype) if coll == "reducescatter" else None)
    for r in range(P):
        assert same_bits(res[r], want[r], dtype), (coll, algo, dtype, op, mode, P, n, r)


# 1,100,007 elements of a 4-byte type over 8 ranks put 537 KB in each
# segment: many blocks per segment on the device path, the persistent grid
# of the host-buffer path
SIZES = (37, 4099, 1100007)


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("coll", ["allreduce", "reducescatter", "allgather"])
def test_host_buffers_match_oracle(coll, dtype, mode):
    for algo, P, pin in (("ring", 8, 1), ("rhd", 5, 1), ("pipeline", 8, 4)):
        for n in SIZES:
            X = hc_inputs.rank_buffers(dtype, P, n, seed=P * 31 + n)
            check_host(coll, algo, X, dtype, "sum", mode, pin)


@pytest.mark.parametrize("mode", ["fused", "step"])
def test_host_buffers_allreduce_ops_hier_and_broadcast(mode):
    for op in ("prod", "max", "min"):
        X = hc_inputs.rank_buffers("float32", 8, 4099, seed=3)
        if op == "prod":
            X = (np.float32(1) + X * np.float32(0.01)).astype(np.float32)
        check_host("allreduce", "rhd", X, "float32", op, mode)
    X = hc_inputs.rank_buffers("bfloat16", 32, 65548, seed=4)
    check_host("allreduce", "hier", X, "bfloat16", "sum", mode, p_intra=8)
    X = hc_inputs.rank_buffers("float32", 6, 1100007, seed=5)
    for root in (0, 3):
        check_host("broadcast", "rhd", X, "float32", "sum", mode, root=root)


def test_host_inputs_device_outputs():
    """Mixed placement: inputs in pinned host memory, outputs in device memory."""
    X = hc_inputs.rank_buffers("float32", 8, 1100007, seed=6)
    check_host("allreduce", "ring", X, "float32", "sum", "fused", recv_on_device=True)
    check_host("allgather", "ring", X, "float32", "sum", "fused", recv_on_device=True)


def test_host_buffers_refuse_pageable_memory():
    """Pageable host memory fails validation with HC_ERR_INVALID_ARG and
    nothing is launched; the same call without host_buffers on device
    memory still works afterwards."""
    from collective_communication_algorithms_gb300 import _binding as B
    P, n = 4, 1024
    pageable = torch.zeros((P, n), dtype=torch.float32)
    assert not pageable.is_pinned()
    dev = torch.ones((P, n), dtype=torch.float32, device="cuda")
    out = torch.empty((P, n), dtype=torch.float32, device="cuda")
    opts = B.make_opts("fused", host_buffers=True)
    with pytest.raises(B.HcError) as e:
        B.hc_allreduce([pageable[r].data_ptr() for r in range(P)],
                       [out[r].data_ptr() for r in range(P)], P, n, "float32", "sum", "ring",
                       opts, 0)
    assert e.value.status == 1
    with pytest.raises(B.HcError) as e:
        B.hc_allreduce([dev[r].data_ptr() for r in range(P)],
                       [pageable[r].data_ptr() for r in range(P)], P, n, "float32", "sum", "ring",
                       opts, 0)
    assert e.value.status == 1
    assert float(pageable.abs().sum()) == 0.0
    B.hc_allreduce([dev[r].data_ptr() for r in range(P)], [out[r].data_ptr() for r in range(P)],
                   P, n, "float32", "sum", "ring", opts, 0)
    torch.cuda.synchronize()
    assert torch.all(out == P)


def test_tensor_wrappers_accept_pinned_tensors():
    import collective_communication_algorithms_gb300 as hc
    P, n = 8, 65548
    X = hc_inputs.rank_buffers("float32", P, n, seed=7)
    send = [torch.from_numpy(X[r].copy()).pin_memory() for r in range(P)]
    recv = [torch.empty(n, dtype=torch.float32).pin_memory() for _ in range(P)]
    hc.allreduce(send, recv, algo="ring")
    torch.cuda.synchronize()
    Y = O.replay("ring", "allreduce", X, "sum", "float32")
    for r in range(P):
        assert same_bits(recv[r].numpy(), Y[r], "float32")
    with pytest.raises(ValueError):
        hc.allreduce([torch.zeros(n) for _ in range(P)])
