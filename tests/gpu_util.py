"""GPU-side helpers for the parity tests: lay P rank buffers out in device
memory (with guard bands), call libhc through its C ABI, read results back.

Every buffer is padded with a guard band filled with a canary pattern; the
helpers return whether any guard element changed, so out-of-bounds writes
fail the test.
"""
import numpy as np
import torch

from collective_communication_algorithms_gb300 import _binding as B

GUARD = 64  # elements of guard band after (and before) each buffer
NP_INT = {"int32": np.int32, "float32": np.int32, "bfloat16": np.int16}
TORCH_INT = {"int32": torch.int32, "float32": torch.int32, "bfloat16": torch.int16}
ESIZE = {"int32": 4, "float32": 4, "bfloat16": 2}
CANARY = {"int32": 0x5A5A5A5A, "float32": 0x5A5A5A5A, "bfloat16": 0x5A5A}


def _as_int(X, dtype):
    return np.ascontiguousarray(X).view(NP_INT[dtype])


class Region:
    """A device buffer of `length` elements with guard bands on both sides,
    16-byte aligned at its first element."""

    def __init__(self, dtype, length, fill_canary=True):
        A = 16 // ESIZE[dtype]
        self.dtype = dtype
        self.length = length
        self.t = torch.empty(GUARD + ((length + A - 1) // A) * A + GUARD, dtype=TORCH_INT[dtype],
                             device="cuda")
        self.t.fill_(np.array(CANARY[dtype]).astype(NP_INT[dtype]).item())
        self.ptr = self.t.data_ptr() + GUARD * ESIZE[dtype]
        assert self.ptr % 16 == 0

    def write(self, arr, at=0):
        a = torch.from_numpy(_as_int(arr, self.dtype).copy()).cuda()
        self.t[GUARD + at:GUARD + at + a.numel()] = a

    def read(self, at=0, length=None):
        length = self.length - at if length is None else length
        return self.t[GUARD + at:GUARD + at + length].cpu().numpy()

    def guards_ok(self):
        h = self.t.cpu().numpy()
        c = np.array(CANARY[self.dtype]).astype(NP_INT[self.dtype])
        pad_end = len(h) - GUARD
        tail = h[GUARD + self.length:]
        return bool(np.all(h[:GUARD] == c) and np.all(tail == c)) and pad_end >= GUARD + self.length


def segments(algo, coll, P, n, dtype):
    return [B.hc_segment_range(algo, coll, P, n, dtype, k)
            for k in range(B.hc_num_segments(algo, coll, P))]


def run_collective(coll, algo, X, dtype, op="sum", mode="fused", in_place=False, p_intra=1,
                   loop_bytes=0, stream=0, root=0):
    """Run one collective through the C ABI on rank vectors X (P, n).
    Returns (results, guards_ok): results[r] is rank r's output (AR/AG: n
    elements; RS: its segment)."""
    P, n = X.shape
    if coll == "broadcast":
        return _run_broadcast(algo, X, dtype, mode, in_place, root, stream)
    segs = segments(algo, coll, P, n, dtype) if coll != "allreduce" else None
    regions = []
    send_ptrs, recv_ptrs = [], []
    scratch = None
    if coll == "allreduce":
        for r in range(P):
            s = Region(dtype, n)
            s.write(X[r])
            regions.append(s)
            if in_place:
                send_ptrs.append(s.ptr)
                recv_ptrs.append(s.ptr)
            else:
                d = Region(dtype, n)
                regions.append(d)
                send_ptrs.append(s.ptr)
                recv_ptrs.append(d.ptr)
        outs = [(regions[r] if in_place else regions[2 * r + 1], 0, n) for r in range(P)]
    elif coll == "reducescatter":
        for r in range(P):
            s = Region(dtype, n)
            s.write(X[r])
            regions.append(s)
            send_ptrs.append(s.ptr)
            off, ln = segs[r]
            if in_place:
                recv_ptrs.append(s.ptr + off * ESIZE[dtype])
            else:
                d = Region(dtype, max(ln, 0))
                regions.append(d)
                recv_ptrs.append(d.ptr)
        if in_place:
            outs = [(regions[r], segs[r][0], segs[r][1]) for r in range(P)]
        else:
            outs = [(regions[2 * r + 1], 0, segs[r][1]) for r in range(P)]
        if mode == "step" and not in_place:
            nbytes = B.hc_scratch_bytes(algo, P, n, dtype)
            scratch = Region("int32", (nbytes + 3) // 4)
    else:
        for r in range(P):
            d = Region(dtype, n)
            regions.append(d)
            recv_ptrs.append(d.ptr)
            off, ln = segs[r]
            if in_place:
                d.write(X[r, off:off + ln], at=off)
                send_ptrs.append(d.ptr + off * ESIZE[dtype])
            else:
                s = Region(dtype, ln)
                s.write(X[r, off:off + ln])
                regions.append(s)
                send_ptrs.append(s.ptr)
        outs = [(regions[r] if in_place else regions[2 * r], 0, n) for r in range(P)]
    opts = B.make_opts(mode, ranks_per_server=p_intra, max_loop_bytes=loop_bytes,
                       scratch=scratch.ptr if scratch else 0,
                       scratch_bytes=(scratch.length * 4) if scratch else 0)
    torch.cuda.synchronize()
    if coll == "allreduce":
        B.hc_allreduce(send_ptrs, recv_ptrs, P, n, dtype, op, algo, opts, stream)
    elif coll == "reducescatter":
        B.hc_reduce_scatter(send_ptrs, recv_ptrs, P, n, dtype, op, algo, opts, stream)
    else:
        B.hc_allgather(send_ptrs, recv_ptrs, P, n, dtype, algo, opts, stream)
    torch.cuda.synchronize()
    res = [reg.read(at, ln) for reg, at, ln in outs]
    ok = all(r.guards_ok() for r in regions) and (scratch is None or scratch.guards_ok())
    return res, ok


def expected(coll, Y, segs):
    """Oracle replay Y (P, n) -> per-rank expected outputs."""
    P = Y.shape[0]
    if coll == "reducescatter":
        return [Y[r, segs[r][0]:segs[r][0] + segs[r][1]] for r in range(P)]
    return [Y[r] for r in range(P)]


def same_bits(a, b, dtype):
    return np.array_equal(_as_int(a, dtype), _as_int(b, dtype))


def _run_broadcast(algo, X, dtype, mode, in_place, root, stream):
    P, n = X.shape
    regions = [Region(dtype, n) for _ in range(P)]
    send = 0
    if in_place:
        regions[root].write(X[root])
    else:
        src = Region(dtype, n)
        src.write(X[root])
        regions.append(src)
        send = src.ptr
    opts = B.make_opts(mode)
    torch.cuda.synchronize()
    B.hc_broadcast(send, [regions[r].ptr for r in range(P)], P, n, dtype, root, algo, opts, stream)
    torch.cuda.synchronize()
    res = [regions[r].read(0, n) for r in range(P)]
    return res, all(r.guards_ok() for r in regions)
