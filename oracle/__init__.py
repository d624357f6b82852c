"""Python view of the C oracle (ctypes + numpy).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py`` may import this package.
The product library (``collective_communication_algorithms_gb300``) never
imports it, and this package never imports the product.

Names follow the pages: algorithms "ring", "rhd", "pipeline"; collectives
"allreduce", "reducescatter", "allgather"; dtypes "int32", "float32",
"bfloat16" (bf16 values travel as numpy uint16 bit patterns); ops "sum",
"prod", "max", "min".
"""
import ctypes
import os

import numpy as np

from . import build as _build

ALGOS = {"ring": 0, "rhd": 1, "pipeline": 2, "hier": 3}
COLLS = {"allreduce": 0, "reducescatter": 1, "allgather": 2, "broadcast": 3}
DTYPES = {"int32": 0, "float32": 1, "bfloat16": 2}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3}
NP_DTYPE = {"int32": np.int32, "float32": np.float32, "bfloat16": np.uint16}
ESIZE = {"int32": 4, "float32": 4, "bfloat16": 2}
MAX_P = 256
SYM_POISON = MAX_P
REDUCE, COPY = 0, 1


class _Msg(ctypes.Structure):
    _fields_ = [("loop", ctypes.c_int32), ("step", ctypes.c_int32),
                ("kind", ctypes.c_int32), ("src", ctypes.c_int32),
                ("dst", ctypes.c_int32), ("seg", ctypes.c_int32),
                ("lo", ctypes.c_int64), ("hi", ctypes.c_int64)]


MSG_DTYPE = np.dtype([("loop", np.int32), ("step", np.int32), ("kind", np.int32),
                      ("src", np.int32), ("dst", np.int32), ("seg", np.int32),
                      ("lo", np.int64), ("hi", np.int64)])

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        L.orc_num_segments.argtypes = [i32, i32, i32, i32]
        L.orc_num_segments.restype = i32
        L.orc_seg_stride.argtypes = [i32, i32, i32, i32, i64, i32]
        L.orc_seg_stride.restype = i64
        L.orc_segment.argtypes = [i32, i32, i32, i32, i64, i32, i32,
                                  ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.orc_segment.restype = i32
        L.orc_slicer.argtypes = [i32, i32, i32, i32, i64, i32, i64,
                                 ctypes.POINTER(i64), ctypes.POINTER(i32), ctypes.POINTER(i64)]
        L.orc_slicer.restype = i32
        L.orc_schedule.argtypes = [i32, i32, i32, i32, i32, i64, i32, i64,
                                   ctypes.POINTER(ctypes.POINTER(_Msg)),
                                   ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.orc_schedule.restype = i64
        L.orc_free.argtypes = [vp]
        L.orc_free.restype = None
        L.orc_replay.argtypes = [i32, i32, i32, i32, i32, i64, i32, i32, i64, vp, vp, i64, vp]
        L.orc_replay.restype = i32
        L.orc_replay_sym.argtypes = [i32, i32, i32, i32, i32, i64, i32, i64, vp, i64, vp]
        L.orc_replay_sym.restype = i32
        L.orc_sym_reset.argtypes = []
        L.orc_sym_reset.restype = None
        L.orc_sym_string.argtypes = [i64, ctypes.c_char_p, i64]
        L.orc_sym_string.restype = i64
        L.orc_sym_leaves.argtypes = [i64, vp]
        L.orc_sym_leaves.restype = i32
        L.orc_direct.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp]
        L.orc_direct.restype = i32
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def num_segments(algo, coll, P, p_intra=1):
    return lib().orc_num_segments(ALGOS[algo], COLLS[coll], P, p_intra)


def segment(algo, coll, P, n, dtype, k, p_intra=1):
    """(offset, length) of segment k."""
    off, ln = ctypes.c_int64(), ctypes.c_int64()
    rc = lib().orc_segment(ALGOS[algo], COLLS[coll], P, p_intra, n, DTYPES[dtype], k,
                           ctypes.byref(off), ctypes.byref(ln))
    if rc:
        raise ValueError("bad segment index")
    return off.value, ln.value


def segments(algo, coll, P, n, dtype, p_intra=1):
    return [segment(algo, coll, P, n, dtype, k, p_intra)
            for k in range(num_segments(algo, coll, P, p_intra))]


def slicer(algo, coll, P, n, dtype, loop_bytes, p_intra=1):
    """(chunk elements per segment per loop, loops, tail elements)."""
    c, nl, t = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int64()
    lib().orc_slicer(ALGOS[algo], COLLS[coll], P, p_intra, n, DTYPES[dtype], loop_bytes,
                     ctypes.byref(c), ctypes.byref(nl), ctypes.byref(t))
    return c.value, nl.value, t.value


def schedule(algo, coll, P, n, dtype="float32", loop_bytes=0, p_intra=1, root=0):
    """Message list (numpy structured array, MSG_DTYPE), steps per loop, loops.
    root is used by the broadcast only."""
    ptr = ctypes.POINTER(_Msg)()
    spl, nl = ctypes.c_int32(), ctypes.c_int32()
    m = lib().orc_schedule(ALGOS[algo], COLLS[coll], P, p_intra, root, n, DTYPES[dtype], loop_bytes,
                           ctypes.byref(ptr), ctypes.byref(spl), ctypes.byref(nl))
    if m < 0:
        raise ValueError("bad schedule arguments")
    try:
        if m > 0:
            raw = ctypes.string_at(ptr, m * ctypes.sizeof(_Msg))
            arr = np.frombuffer(raw, dtype=MSG_DTYPE).copy()
        else:
            arr = np.zeros(0, dtype=MSG_DTYPE)
    finally:
        lib().orc_free(ptr)
    return arr, spl.value, nl.value


def _check_X(X, dtype):
    X = np.ascontiguousarray(X)
    if X.ndim != 2 or X.dtype != NP_DTYPE[dtype]:
        raise TypeError("X must be a (P, n) array of %s" % NP_DTYPE[dtype])
    return X


def replay(algo, coll, X, op, dtype, loop_bytes=0, p_intra=1, J=None, root=0):
    """Step-by-step replay of the schedule on rank vectors X (P, n).

    Returns (P, len(J)) values after the schedule (J = all elements by default):
    for allreduce every row is that rank's output; for reducescatter rank r's
    result is its row restricted to segment r; for allgather every row is the
    gathered vector; for broadcast every row is the root's vector.
    """
    X = _check_X(X, dtype)
    P, n = X.shape
    if J is None:
        Jp, nJ = None, n
    else:
        J = np.ascontiguousarray(J, dtype=np.int64)
        Jp, nJ = J.ctypes.data, J.size
    Y = np.empty((P, nJ), dtype=NP_DTYPE[dtype])
    rc = lib().orc_replay(ALGOS[algo], COLLS[coll], P, p_intra, root, n, DTYPES[dtype], OPS[op],
                          loop_bytes, X.ctypes.data, Jp, nJ, Y.ctypes.data)
    if rc:
        raise ValueError("oracle replay rejected its arguments")
    return Y


def replay_sym(algo, coll, P, n, layout_dtype="float32", loop_bytes=0, p_intra=1, J=None, root=0):
    """Symbolic replay: (P, len(J)) int64 expression node ids."""
    if J is None:
        Jp, nJ = None, n
    else:
        J = np.ascontiguousarray(J, dtype=np.int64)
        Jp, nJ = J.ctypes.data, J.size
    Y = np.empty((P, nJ), dtype=np.int64)
    rc = lib().orc_replay_sym(ALGOS[algo], COLLS[coll], P, p_intra, root, n, DTYPES[layout_dtype],
                              loop_bytes, Jp, nJ, Y.ctypes.data)
    if rc:
        raise ValueError("oracle symbolic replay rejected its arguments")
    return Y


def sym_reset():
    lib().orc_sym_reset()


def sym_string(node):
    need = lib().orc_sym_string(int(node), None, 0)
    buf = ctypes.create_string_buffer(int(need) + 1)
    lib().orc_sym_string(int(node), buf, need + 1)
    return buf.value.decode()


def sym_leaves(node):
    """Leaf multiplicities: array of MAX_P + 1 counts (last = never written)."""
    counts = np.zeros(MAX_P + 1, dtype=np.int64)
    if lib().orc_sym_leaves(int(node), counts.ctypes.data):
        raise MemoryError
    return counts


def direct(X, op, dtype):
    """Straight from the definition Y[j] = (+)_i X_i[j].

    Returns (raw, f64, abs_sum): raw bits for int32 and for max/min (None for
    fp sum/prod), the binary64 value for sum/prod (None for max/min), and
    sum_i |X_i[j]| in binary64 for fp sum (else None).
    """
    X = _check_X(X, dtype)
    P, n = X.shape
    raw = np.zeros(n, dtype=NP_DTYPE[dtype])
    y64 = np.zeros(n, dtype=np.float64)
    s1 = np.zeros(n, dtype=np.float64)
    rc = lib().orc_direct(DTYPES[dtype], OPS[op], P, n, X.ctypes.data, raw.ctypes.data,
                          y64.ctypes.data, s1.ctypes.data)
    if rc:
        raise ValueError("bad direct arguments")
    is_fp = dtype != "int32"
    if op in ("max", "min"):
        return raw, None, None
    if is_fp:
        return None, y64, (s1 if op == "sum" else None)
    return raw, y64, None


def f32_to_bf16(x: float) -> int:
    return int(lib().orc_f32_to_bf16(ctypes.c_float(x)))

