"""The bounded waits of the TMA-staged kernels, made to run out on purpose.

Every wait of a libhc kernel on a shared-memory barrier gives up after a
limit, records HC_ERR_TIMEOUT in a device flag that hc_device_status reads
and clears, and lets the block exit once its own bulk copies have landed.
hc_test_expire_waits(1) arms that path without any fault: the barrier
expects one arrival more than the block makes before its first wait, whose
limit drops to 1 ms, so that wait expires although every copy lands; the
block then records the timeout, makes the held arrival, waits for its copies
and exits.  These tests check, for the fused AllReduce / ReduceScatter
(fused_reduce_tma) and the TMA-staged step kernel (step_kernel_tma: the
Pipeline's mesh reduce, and its AllGather steps' broadcasts by bulk
stores), that

  * the call completes, well inside the 2 s normal limit (no second wait
    ran out: the held arrival released the barrier),
  * nothing was written outside the output buffers (guard bands),
  * hc_device_status() reports HC_ERR_TIMEOUT, clears it on request, and
    reports HC_OK afterwards,
  * the next call, with the mode switched off, is bit-exact against the
    oracle.
"""
import time

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
from gpu_util import expected, run_collective, same_bits, segments  # noqa: E402

HC_OK, HC_ERR_TIMEOUT = 0, 6

# (collective, algo, mode, P, n, ranks_per_server): each case runs a
# TMA-staged kernel -- the step-mode Pipeline AllReduce starts with a mesh
# reduce of 4 inputs, and every launch of the step-mode Pipeline AllGather
# (2 servers of 4) copies each block to 4 ranks by bulk stores
CASES = [
    ("allreduce", "ring", "fused", 8, 40003, 1),
    ("reducescatter", "rhd", "fused", 12, 30011, 1),
    ("allreduce", "pipeline", "step", 8, 20011, 4),
    ("allgather", "pipeline", "step", 8, 8 * 20011 + 5, 4),
]


@pytest.mark.parametrize("coll,algo,mode,P,n,rps", CASES)
def test_expired_wait_reports_timeout_then_recovers(coll, algo, mode, P, n, rps):
    X = hc_inputs.gradients_f32(P, n, seed=P + n)
    # load the kernels first, so module loading is not timed below
    run_collective(coll, algo, X, "float32", "sum", mode, p_intra=rps)
    assert B.hc_device_status(clear=True) == HC_OK
    B.hc_test_expire_waits(True)
    try:
        t0 = time.perf_counter()
        _, ok = run_collective(coll, algo, X, "float32", "sum", mode, p_intra=rps)
        elapsed = time.perf_counter() - t0
    finally:
        B.hc_test_expire_waits(False)
    assert ok, "a block wrote outside its buffers"
    assert elapsed < 1.0, elapsed  # each block's first wait: 1 ms; no 2 s wait ran out
    assert B.hc_device_status(clear=False) == HC_ERR_TIMEOUT
    assert B.hc_device_status(clear=True) == HC_ERR_TIMEOUT
    assert B.hc_device_status(clear=False) == HC_OK
    # normal operation again: bit-exact against the oracle, no timeout
    res, ok = run_collective(coll, algo, X, "float32", "sum", mode, p_intra=rps)
    assert ok
    Y = O.replay(algo, coll, X, "sum", "float32", p_intra=rps)
    segs = segments(algo, coll, P, n, "float32") if coll != "allreduce" else None
    for r, (got, want) in enumerate(zip(res, expected(coll, Y, segs))):
        assert same_bits(got, want, "float32"), (coll, algo, mode, r)
    assert B.hc_device_status(clear=False) == HC_OK
