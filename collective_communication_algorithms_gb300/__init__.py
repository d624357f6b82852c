"""GB300-native data plane of HCCL-style AllReduce / ReduceScatter /
AllGather schedules (Ring, Recursive Halving-Doubling, hierarchical
Pipeline) for P virtual ranks whose buffers live in one GPU's memory.

The work happens in libhc (include/hc.h), hand-written sm_103a kernels behind
a C ABI.  This package is its thin Python binding: the hc_* functions mirror
the C entry points; allreduce / reduce_scatter / allgather / broadcast accept
lists of torch tensors (one per virtual rank: CUDA tensors, or pinned host
tensors that the kernels then read and write over the host link) and pass
their pointers and the current CUDA stream.  PyTorch only provides device memory and streams.
"""
from ._binding import (ALGOS, COLLS, DTYPES, MODES, OPS, Graph, HcError, hc_allgather, hc_allreduce,
                       hc_broadcast,
                       hc_num_segments, hc_reduce_scatter, hc_schedule_stats, hc_scratch_bytes,
                       hc_segment_range, hc_step_plan, hc_version, lib, make_opts)
from ._binding import LIB_PATH as library_path

__all__ = ["allreduce", "reduce_scatter", "allgather", "broadcast", "segment_range", "segments",
           "Graph", "hc_broadcast",
           "hc_allreduce", "hc_reduce_scatter", "hc_allgather", "hc_segment_range",
           "hc_num_segments", "hc_scratch_bytes", "hc_schedule_stats", "hc_step_plan",
           "hc_version", "HcError", "make_opts", "library_path", "lib"]

_TORCH_DTYPE = {"torch.int32": "int32", "torch.float32": "float32", "torch.bfloat16": "bfloat16"}


def _dtype_name(t):
    name = _TORCH_DTYPE.get(str(t.dtype))
    if name is None:
        raise TypeError("unsupported dtype %s (int32, float32, bfloat16)" % t.dtype)
    return name


def _stream(stream):
    if stream is not None:
        return int(getattr(stream, "cuda_stream", stream))
    import torch
    return int(torch.cuda.current_stream().cuda_stream)


def _ptrs(ts):
    for t in ts:
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError("rank buffers must be contiguous CUDA or pinned host tensors")
    return [t.data_ptr() for t in ts]


def _on_host(*groups):
    """True when some rank buffer is a pinned host tensor: the kernels then
    read or write it over the host link (hc_opts_t.host_buffers)."""
    return any(not t.is_cuda for g in groups if g is not None for t in g)


def segment_range(algo, coll, P, count, dtype, k):
    return hc_segment_range(algo, coll, P, count, dtype, k)


def segments(algo, coll, P, count, dtype):
    return [hc_segment_range(algo, coll, P, count, dtype, k)
            for k in range(hc_num_segments(algo, coll, P))]


def _opts(mode, ranks_per_server, max_loop_bytes, scratch, host=False):
    sp, sb = 0, 0
    if scratch is not None:
        sp, sb = scratch.data_ptr(), scratch.numel() * scratch.element_size()
    return make_opts(mode, ranks_per_server, max_loop_bytes, sp, sb, host_buffers=host)


def allreduce(send, recv=None, op="sum", algo="ring", mode="fused", ranks_per_server=1,
              max_loop_bytes=0, stream=None):
    """recv[r] = (+)_i send[i]; recv=None means in place."""
    recv = send if recv is None else recv
    P = len(send)
    hc_allreduce(_ptrs(send), _ptrs(recv), P, send[0].numel(), _dtype_name(send[0]), op, algo,
                 _opts(mode, ranks_per_server, max_loop_bytes, None, _on_host(send, recv)),
                 _stream(stream))
    return recv


def reduce_scatter(send, recv, op="sum", algo="ring", mode="fused", ranks_per_server=1,
                   max_loop_bytes=0, scratch=None, stream=None):
    """recv[r] = segment r of (+)_i send[i] (see segments())."""
    P = len(send)
    hc_reduce_scatter(_ptrs(send), _ptrs(recv), P, send[0].numel(), _dtype_name(send[0]), op,
                      algo, _opts(mode, ranks_per_server, max_loop_bytes, scratch,
                                  _on_host(send, recv)),
                      _stream(stream))
    return recv


def allgather(send, recv, algo="ring", mode="fused", ranks_per_server=1, max_loop_bytes=0,
              stream=None):
    """recv[r][segment k] = send[k]; send=None means in place."""
    P = len(recv)
    hc_allgather(None if send is None else _ptrs(send), _ptrs(recv), P, recv[0].numel(),
                 _dtype_name(recv[0]), algo,
                 _opts(mode, ranks_per_server, max_loop_bytes, None, _on_host(send, recv)),
                 _stream(stream))
    return recv


def broadcast(send, recv, root=0, algo="rhd", mode="fused", stream=None):
    """recv[r] = send (the root's vector) for every rank; send=None: in place
    from recv[root]."""
    P = len(recv)
    if send is not None:
        _ptrs([send])
    hc_broadcast(None if send is None else send.data_ptr(), _ptrs(recv), P, recv[0].numel(),
                 _dtype_name(recv[0]), root, algo,
                 _opts(mode, 1, 0, None, _on_host(None if send is None else [send], recv)),
                 _stream(stream))
    return recv
