"""ctypes binding of libhc (include/hc.h).  Argument marshalling only: every
step of every collective runs in libhc's CUDA kernels.

The functions named hc_* take raw values exactly like the C entry points
(device pointers as ints, a stream handle as an int) and raise HcError on a
non-zero status.  There is no fallback: if libhc.so was not built, loading it
raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libhc.so")
MAX_RANKS = 64

DTYPES = {"int32": 0, "float32": 1, "bfloat16": 2}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3}
ALGOS = {"ring": 0, "rhd": 1, "pipeline": 2, "hier": 3}
COLLS = {"allreduce": 0, "reducescatter": 1, "allgather": 2, "broadcast": 3}
MODES = {"fused": 0, "step": 1}
STATUS = {0: "HC_OK", 1: "HC_ERR_INVALID_ARG", 2: "HC_ERR_UNSUPPORTED", 3: "HC_ERR_ALIGN",
          4: "HC_ERR_SCRATCH", 5: "HC_ERR_CUDA", 6: "HC_ERR_TIMEOUT"}


class HcError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        self.name = STATUS.get(status, str(status))
        detail = status_string(status)
        if status == 5:
            try:
                detail += ", " + lib().hc_last_cuda_error().decode()
            except Exception:
                pass
        super().__init__("%s: %s (%s)" % (where, self.name, detail))


class hc_opts_t(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("mode", ctypes.c_int),
                ("ranks_per_server", ctypes.c_int), ("max_loop_bytes", ctypes.c_size_t),
                ("scratch", ctypes.c_void_p), ("scratch_bytes", ctypes.c_size_t),
                ("host_buffers", ctypes.c_int)]


class hc_stats_t(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("steps_per_loop", ctypes.c_int),
                ("loops", ctypes.c_int), ("chunk", ctypes.c_size_t), ("tail", ctypes.c_size_t),
                ("launches_step", ctypes.c_int), ("launches_fused", ctypes.c_int),
                ("step_bytes", ctypes.c_ulonglong), ("fused_bytes", ctypes.c_ulonglong)]


class hc_plan_record_t(ctypes.Structure):
    _fields_ = [("launch", ctypes.c_int32), ("seg", ctypes.c_int32),
                ("lo", ctypes.c_int64), ("hi", ctypes.c_int64),
                ("acc_rank", ctypes.c_int32), ("acc_loc", ctypes.c_int32),
                ("in_loc", ctypes.c_int32), ("in_cnt", ctypes.c_int32),
                ("out_loc", ctypes.c_int32), ("out_cnt", ctypes.c_int32),
                ("in_ranks", ctypes.c_int32 * MAX_RANKS),
                ("out_ranks", ctypes.c_int32 * MAX_RANKS)]


# every symbol include/hc.h declares
EXPORTS = ("hc_allreduce", "hc_reduce_scatter", "hc_reduce_scatter_static_scratch",
           "hc_allgather", "hc_broadcast", "hc_segment_range", "hc_graph_create",
           "hc_graph_add_allreduce", "hc_graph_add_reduce_scatter", "hc_graph_add_allgather",
           "hc_graph_add_broadcast", "hc_graph_build",
           "hc_graph_launch", "hc_graph_info", "hc_graph_destroy",
           "hc_num_segments", "hc_scratch_bytes", "hc_schedule_stats", "hc_step_plan",
           "hc_select_algo", "hc_device_status", "hc_test_expire_waits", "hc_last_cuda_error",
           "hc_status_string",
           "hc_version")

_lib = None


def lib():
    """Load libhc.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libhc.so is not built (%s); run "
                               "collective_communication_algorithms_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        ptrs = ctypes.POINTER(ctypes.c_void_p)
        for name in ("hc_allreduce", "hc_reduce_scatter"):
            f = getattr(L, name)
            f.argtypes = [ptrs, ptrs, i32, sz, i32, i32, i32, ctypes.POINTER(hc_opts_t), vp]
            f.restype = i32
        L.hc_reduce_scatter_static_scratch.argtypes = [ptrs, ptrs, i32, sz, i32, i32, i32, i32,
                                                       sz, vp]
        L.hc_reduce_scatter_static_scratch.restype = i32
        L.hc_allgather.argtypes = [ptrs, ptrs, i32, sz, i32, i32, ctypes.POINTER(hc_opts_t), vp]
        L.hc_allgather.restype = i32
        L.hc_graph_create.argtypes = [ctypes.POINTER(vp)]
        L.hc_graph_create.restype = i32
        for name in ("hc_graph_add_allreduce", "hc_graph_add_reduce_scatter"):
            f = getattr(L, name)
            f.argtypes = [vp, ptrs, ptrs, i32, sz, i32, i32, i32, ctypes.POINTER(hc_opts_t)]
            f.restype = i32
        L.hc_graph_add_allgather.argtypes = [vp, ptrs, ptrs, i32, sz, i32, i32,
                                             ctypes.POINTER(hc_opts_t)]
        L.hc_graph_add_allgather.restype = i32
        L.hc_graph_add_broadcast.argtypes = [vp, vp, ptrs, i32, sz, i32, i32, i32,
                                             ctypes.POINTER(hc_opts_t)]
        L.hc_graph_add_broadcast.restype = i32
        L.hc_broadcast.argtypes = [vp, ptrs, i32, sz, i32, i32, i32, ctypes.POINTER(hc_opts_t), vp]
        L.hc_broadcast.restype = i32
        for name in ("hc_graph_build", "hc_graph_destroy"):
            getattr(L, name).argtypes = [vp]
            getattr(L, name).restype = i32
        L.hc_graph_launch.argtypes = [vp, vp]
        L.hc_graph_launch.restype = i32
        L.hc_graph_info.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                    ctypes.POINTER(i32)]
        L.hc_graph_info.restype = i32
        L.hc_segment_range.argtypes = [i32, i32, i32, sz, i32, i32,
                                       ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.hc_segment_range.restype = i32
        L.hc_num_segments.argtypes = [i32, i32, i32]
        L.hc_num_segments.restype = i32
        L.hc_scratch_bytes.argtypes = [i32, i32, sz, i32]
        L.hc_scratch_bytes.restype = sz
        L.hc_schedule_stats.argtypes = [i32, i32, i32, i32, sz, i32, sz,
                                        ctypes.POINTER(hc_stats_t),
                                        ctypes.POINTER(ctypes.c_ulonglong)]
        L.hc_schedule_stats.restype = i32
        L.hc_step_plan.argtypes = [i32, i32, i32, i32, sz, i32, sz, i32, i32,
                                   ctypes.POINTER(hc_plan_record_t), sz,
                                   ctypes.POINTER(sz), ctypes.POINTER(i32)]
        L.hc_step_plan.restype = i32
        L.hc_select_algo.argtypes = [i32, i32, i32, sz, i32, i32, ctypes.POINTER(i32),
                                     ctypes.POINTER(ctypes.c_double)]
        L.hc_select_algo.restype = i32
        L.hc_last_cuda_error.argtypes = []
        L.hc_last_cuda_error.restype = ctypes.c_char_p
        L.hc_device_status.argtypes = [i32]
        L.hc_device_status.restype = i32
        L.hc_test_expire_waits.argtypes = [i32]
        L.hc_test_expire_waits.restype = i32
        L.hc_status_string.argtypes = [i32]
        L.hc_status_string.restype = ctypes.c_char_p
        L.hc_version.argtypes = []
        L.hc_version.restype = i32
        _lib = L
    return _lib


def status_string(status):
    try:
        return lib().hc_status_string(int(status)).decode()
    except Exception:  # library missing: the code alone
        return STATUS.get(status, "?")


def _check(status, where):
    if status != 0:
        raise HcError(status, where)


def _ptr_array(ptrs):
    if ptrs is None or isinstance(ptrs, ctypes.Array):
        return ptrs  # None, or an array built once with ptr_array() and reused
    arr = (ctypes.c_void_p * len(ptrs))()
    for i, p in enumerate(ptrs):
        arr[i] = int(p) if p else None
    return arr


def ptr_array(ptrs):
    """A ctypes array of the pointers, which every hc_* function accepts in
    place of a list: callers that issue many calls on the same buffers build
    it once and skip the per-call conversion."""
    return _ptr_array(list(ptrs))


def make_opts(mode="fused", ranks_per_server=1, max_loop_bytes=0, scratch=0, scratch_bytes=0,
              host_buffers=False):
    o = hc_opts_t()
    o.struct_size = ctypes.sizeof(hc_opts_t)
    o.mode = MODES[mode] if isinstance(mode, str) else int(mode)
    o.ranks_per_server = int(ranks_per_server)
    o.max_loop_bytes = int(max_loop_bytes)
    o.scratch = int(scratch) if scratch else None
    o.scratch_bytes = int(scratch_bytes)
    o.host_buffers = 1 if host_buffers else 0
    return o


def _enum(table, v):
    return table[v] if isinstance(v, str) else int(v)


def hc_allreduce(send, recv, P, count, dtype, op, algo, opts=None, stream=0):
    st = lib().hc_allreduce(_ptr_array(send), _ptr_array(recv), int(P), int(count),
                            _enum(DTYPES, dtype), _enum(OPS, op), _enum(ALGOS, algo),
                            ctypes.byref(opts) if opts is not None else None,
                            ctypes.c_void_p(int(stream)) if stream else None)
    _check(st, "hc_allreduce")


def hc_reduce_scatter(send, recv, P, count, dtype, op, algo, opts=None, stream=0):
    st = lib().hc_reduce_scatter(_ptr_array(send), _ptr_array(recv), int(P), int(count),
                                 _enum(DTYPES, dtype), _enum(OPS, op), _enum(ALGOS, algo),
                                 ctypes.byref(opts) if opts is not None else None,
                                 ctypes.c_void_p(int(stream)) if stream else None)
    _check(st, "hc_reduce_scatter")


class BoundCall:
    """One collective call whose arguments were converted to C types once:
    calling it issues the C entry point again with exactly those arguments
    (same buffers, sizes, options and stream).  For callers that repeat a
    call, e.g. once per training step, this skips the per-call argument
    conversion of the hc_* functions; the status is checked as they do."""

    __slots__ = ("fn", "args", "name", "keep")

    def __init__(self, name, args, keep):
        self.fn = lib()[name]  # a function object of its own, without argument conversion
        self.fn.restype = ctypes.c_int
        self.args = args
        self.name = name
        self.keep = keep  # the objects the arguments point into

    def __call__(self):
        st = self.fn(*self.args)
        if st:
            raise HcError(st, self.name)


def _bound_args(send, recv, P, count, dtype, opts, stream):
    sp, rp = _ptr_array(list(send)) if send is not None else None, _ptr_array(list(recv))
    head = (sp, rp, ctypes.c_int(int(P)), ctypes.c_size_t(int(count)),
            ctypes.c_int(_enum(DTYPES, dtype)))
    tail = (ctypes.byref(opts) if opts is not None else None,
            ctypes.c_void_p(int(stream)) if stream else None)
    return head, tail, (sp, rp, opts)


def bind_allreduce(send, recv, P, count, dtype, op, algo, opts=None, stream=0):
    """hc_allreduce with these arguments, as a BoundCall."""
    head, tail, keep = _bound_args(send, recv, P, count, dtype, opts, stream)
    mid = (ctypes.c_int(_enum(OPS, op)), ctypes.c_int(_enum(ALGOS, algo)))
    return BoundCall("hc_allreduce", head + mid + tail, keep)


def bind_reduce_scatter(send, recv, P, count, dtype, op, algo, opts=None, stream=0):
    """hc_reduce_scatter with these arguments, as a BoundCall."""
    head, tail, keep = _bound_args(send, recv, P, count, dtype, opts, stream)
    mid = (ctypes.c_int(_enum(OPS, op)), ctypes.c_int(_enum(ALGOS, algo)))
    return BoundCall("hc_reduce_scatter", head + mid + tail, keep)


def bind_allgather(send, recv, P, count, dtype, algo, opts=None, stream=0):
    """hc_allgather with these arguments, as a BoundCall."""
    head, tail, keep = _bound_args(send, recv, P, count, dtype, opts, stream)
    return BoundCall("hc_allgather", head + (ctypes.c_int(_enum(ALGOS, algo)),) + tail, keep)


def hc_reduce_scatter_static_scratch(send, recv, P, count, dtype, op, algo, ranks_per_server=1,
                                     max_loop_bytes=0, stream=0):
    """Step-mode ReduceScatter whose working memory is the library's own
    fixed device array (for callers that may not allocate device memory)."""
    st = lib().hc_reduce_scatter_static_scratch(
        _ptr_array(send), _ptr_array(recv), int(P), int(count), _enum(DTYPES, dtype),
        _enum(OPS, op), _enum(ALGOS, algo), int(ranks_per_server), int(max_loop_bytes),
        ctypes.c_void_p(int(stream)) if stream else None)
    _check(st, "hc_reduce_scatter_static_scratch")


def hc_allgather(send, recv, P, count, dtype, algo, opts=None, stream=0):
    st = lib().hc_allgather(_ptr_array(send), _ptr_array(recv), int(P), int(count),
                            _enum(DTYPES, dtype), _enum(ALGOS, algo),
                            ctypes.byref(opts) if opts is not None else None,
                            ctypes.c_void_p(int(stream)) if stream else None)
    _check(st, "hc_allgather")


def hc_broadcast(send, recv, P, count, dtype, root, algo="rhd", opts=None, stream=0):
    """send: device pointer of the root's vector, or 0/None for in place."""
    st = lib().hc_broadcast(ctypes.c_void_p(int(send)) if send else None, _ptr_array(recv), int(P),
                            int(count), _enum(DTYPES, dtype), int(root), _enum(ALGOS, algo),
                            ctypes.byref(opts) if opts is not None else None,
                            ctypes.c_void_p(int(stream)) if stream else None)
    _check(st, "hc_broadcast")


def hc_segment_range(algo, coll, P, count, dtype, k):
    off, ln = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().hc_segment_range(_enum(ALGOS, algo), _enum(COLLS, coll), int(P), int(count),
                                  _enum(DTYPES, dtype), int(k), ctypes.byref(off),
                                  ctypes.byref(ln)), "hc_segment_range")
    return off.value, ln.value


def hc_num_segments(algo, coll, P):
    return lib().hc_num_segments(_enum(ALGOS, algo), _enum(COLLS, coll), int(P))


def hc_scratch_bytes(algo, P, count, dtype):
    return lib().hc_scratch_bytes(_enum(ALGOS, algo), int(P), int(count), _enum(DTYPES, dtype))


def hc_schedule_stats(algo, coll, P, count, dtype, ranks_per_server=1, max_loop_bytes=0):
    """Returns (stats dict, per-rank bytes sent list)."""
    s = hc_stats_t()
    s.struct_size = ctypes.sizeof(hc_stats_t)
    sent = (ctypes.c_ulonglong * int(P))()
    _check(lib().hc_schedule_stats(_enum(ALGOS, algo), _enum(COLLS, coll), int(P),
                                   int(ranks_per_server), int(count), _enum(DTYPES, dtype),
                                   int(max_loop_bytes), ctypes.byref(s), sent),
           "hc_schedule_stats")
    d = {name: getattr(s, name) for name, _ in hc_stats_t._fields_ if name != "struct_size"}
    return d, list(sent)


def hc_step_plan(algo, coll, P, count, dtype, ranks_per_server=1, max_loop_bytes=0,
                 in_place=True, root=0):
    """Returns (list of record dicts, number of launches)."""
    L = lib()
    n = ctypes.c_size_t()
    nl = ctypes.c_int()
    args = (_enum(ALGOS, algo), _enum(COLLS, coll), int(P), int(ranks_per_server), int(count),
            _enum(DTYPES, dtype), int(max_loop_bytes), 1 if in_place else 0, int(root))
    _check(L.hc_step_plan(*args, None, 0, ctypes.byref(n), ctypes.byref(nl)), "hc_step_plan")
    recs = (hc_plan_record_t * max(1, n.value))()
    _check(L.hc_step_plan(*args, recs, n.value, ctypes.byref(n), ctypes.byref(nl)),
           "hc_step_plan")
    out = []
    for i in range(n.value):
        r = recs[i]
        out.append({"launch": r.launch, "seg": r.seg, "lo": r.lo, "hi": r.hi,
                    "acc_rank": r.acc_rank, "acc_loc": r.acc_loc, "in_loc": r.in_loc,
                    "out_loc": r.out_loc,
                    "in_ranks": list(r.in_ranks[:r.in_cnt]),
                    "out_ranks": list(r.out_ranks[:r.out_cnt])})
    return out, nl.value


def hc_select_algo(coll, P, count, dtype, mode="step", ranks_per_server=1):
    """(algorithm name, predicted microseconds) of the cost model."""
    a, t = ctypes.c_int(), ctypes.c_double()
    _check(lib().hc_select_algo(_enum(COLLS, coll), int(P), int(ranks_per_server), int(count),
                                _enum(DTYPES, dtype), _enum(MODES, mode), ctypes.byref(a),
                                ctypes.byref(t)), "hc_select_algo")
    name = {v: k for k, v in ALGOS.items()}[a.value]
    return name, t.value


def hc_device_status(clear=True):
    """HC_OK (0) or HC_ERR_TIMEOUT (6) recorded by a bounded device-side wait."""
    return lib().hc_device_status(1 if clear else 0)


class Graph:
    """Graph mode: collectives added once, replayed with one launch."""

    def __init__(self):
        self.handle = ctypes.c_void_p()
        _check(lib().hc_graph_create(ctypes.byref(self.handle)), "hc_graph_create")

    def add_allreduce(self, send, recv, P, count, dtype, op, algo, opts=None):
        _check(lib().hc_graph_add_allreduce(self.handle, _ptr_array(send), _ptr_array(recv),
                                            int(P), int(count), _enum(DTYPES, dtype),
                                            _enum(OPS, op), _enum(ALGOS, algo),
                                            ctypes.byref(opts) if opts is not None else None),
               "hc_graph_add_allreduce")

    def add_reduce_scatter(self, send, recv, P, count, dtype, op, algo, opts=None):
        _check(lib().hc_graph_add_reduce_scatter(self.handle, _ptr_array(send),
                                                 _ptr_array(recv), int(P), int(count),
                                                 _enum(DTYPES, dtype), _enum(OPS, op),
                                                 _enum(ALGOS, algo),
                                                 ctypes.byref(opts) if opts is not None else None),
               "hc_graph_add_reduce_scatter")

    def add_allgather(self, send, recv, P, count, dtype, algo, opts=None):
        _check(lib().hc_graph_add_allgather(self.handle, _ptr_array(send), _ptr_array(recv),
                                            int(P), int(count), _enum(DTYPES, dtype),
                                            _enum(ALGOS, algo),
                                            ctypes.byref(opts) if opts is not None else None),
               "hc_graph_add_allgather")

    def add_broadcast(self, send, recv, P, count, dtype, root, algo="rhd", opts=None):
        _check(lib().hc_graph_add_broadcast(self.handle, ctypes.c_void_p(int(send)) if send else None,
                                            _ptr_array(recv), int(P), int(count),
                                            _enum(DTYPES, dtype), int(root), _enum(ALGOS, algo),
                                            ctypes.byref(opts) if opts is not None else None),
               "hc_graph_add_broadcast")

    def build(self):
        _check(lib().hc_graph_build(self.handle), "hc_graph_build")

    def launch(self, stream=0):
        _check(lib().hc_graph_launch(self.handle, ctypes.c_void_p(int(stream)) if stream else None),
               "hc_graph_launch")

    def info(self):
        a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(lib().hc_graph_info(self.handle, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "hc_graph_info")
        return {"collectives": a.value, "edges": b.value, "kernels": c.value}

    def close(self):
        if self.handle:
            lib().hc_graph_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hc_test_expire_waits(enable):
    """Test hook: TMA-staged kernels (fused and step) launched while enabled
    give up their first shared-memory barrier wait after 1 ms and report
    HC_ERR_TIMEOUT."""
    _check(lib().hc_test_expire_waits(1 if enable else 0), "hc_test_expire_waits")


def hc_version():
    return lib().hc_version()
