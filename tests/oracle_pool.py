"""Whole-vector oracle replays at the benchmark sizes, spread over the host
cores (test infrastructure).

The oracle replays a schedule on any sorted set of element indices, so a
vector of n elements per rank splits into contiguous windows of indices that
separate processes replay independently: every element's value depends only
on the same element of the P rank vectors.  The rank vectors X (P, n) and the
result Y (P, n) sit in memory-mapped files that every worker maps; a worker
replays window [lo, hi) and writes Y[:, lo:hi].  Workers are spawned, never
forked, so that a parent that has initialised CUDA is safe.

Nothing here computes anything of the method itself: every value comes from
oracle.replay.
"""
import os
import shutil
import tempfile
from concurrent.futures import ProcessPoolExecutor
import multiprocessing as mp

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CELLS_PER_WINDOW = 1 << 23  # P x window elements of replay state per worker task


def _replay_window(task):
    (xpath, ypath, shape, dtype_str, algo, coll, op, dtype, p_intra, loop_bytes, root, lo, hi) = task
    import oracle as O
    X = np.memmap(xpath, dtype=np.dtype(dtype_str), mode="r", shape=shape)
    Y = np.memmap(ypath, dtype=np.dtype(dtype_str), mode="r+", shape=shape)
    J = np.arange(lo, hi, dtype=np.int64)
    Y[:, lo:hi] = O.replay(algo, coll, np.asarray(X), op, dtype, loop_bytes=loop_bytes,
                           p_intra=p_intra, J=J, root=root)
    Y.flush()
    del X, Y
    return hi - lo


def _scratch_dir(need_bytes):
    """A directory with room for the two mapped files: shared memory if it
    has the room, else the system's temporary directory, else the repo."""
    for d in ("/dev/shm", tempfile.gettempdir(), ROOT):
        try:
            st = os.statvfs(d)
            if st.f_bavail * st.f_frsize > 1.25 * need_bytes and os.access(d, os.W_OK):
                return tempfile.mkdtemp(prefix="hc_oracle_", dir=d)
        except OSError:
            continue
    raise RuntimeError("no room for %d bytes of oracle state" % need_bytes)


class OraclePool:
    """A pool of spawned oracle workers, one per host core (at most 16)."""

    def __init__(self, workers=None):
        self.workers = workers or max(1, min(16, os.cpu_count() or 1))
        self.ex = ProcessPoolExecutor(max_workers=self.workers, mp_context=mp.get_context("spawn"))

    def close(self):
        self.ex.shutdown(wait=True)

    def replay(self, algo, coll, X, op, dtype, loop_bytes=0, p_intra=1, root=0):
        """oracle.replay(algo, coll, X, op, dtype, ...) over all n elements,
        computed window by window in the workers: a (P, n) array."""
        X = np.ascontiguousarray(X)
        P, n = X.shape
        d = _scratch_dir(2 * X.nbytes)
        try:
            xpath, ypath = os.path.join(d, "x.bin"), os.path.join(d, "y.bin")
            Xm = np.memmap(xpath, dtype=X.dtype, mode="w+", shape=X.shape)
            Xm[:] = X
            Xm.flush()
            del Xm
            Ym = np.memmap(ypath, dtype=X.dtype, mode="w+", shape=X.shape)
            del Ym
            w = max(64, CELLS_PER_WINDOW // P)
            tasks = [(xpath, ypath, X.shape, X.dtype.str, algo, coll, op, dtype, p_intra,
                      loop_bytes, root, lo, min(n, lo + w)) for lo in range(0, n, w)]
            done = sum(self.ex.map(_replay_window, tasks))
            assert done == n
            return np.array(np.memmap(ypath, dtype=X.dtype, mode="r", shape=X.shape))
        finally:
            shutil.rmtree(d, ignore_errors=True)
