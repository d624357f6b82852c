"""The multi-GPU benchmark runs independent replicas: one process per GPU,
each doing the whole collective on its own buffers, with no data-path
exchange.  The host logic that joins them (barrier, maximum of the ranks'
times, whole-job algbw = N x per-rank bytes / slowest time) runs here as two
gloo ranks on the CPU, and the reference arm's ranks other than 0 must exit
without work."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method="tcp://127.0.0.1:%d" % port)
    try:
        # rank r took (r + 1) ms in total and 0.5 / (r + 1) ms per kernel
        got = bench.max_over_ranks([rank + 1.0, 0.5 / (rank + 1)], world, "cpu")
        dist.barrier()
        out.put((rank, got, bench.replica_algbw(world, 64 << 20, got[0])))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (g, v)) for r, g, v in (q.get(timeout=120) for _ in range(world)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        got, value = res[r]
        assert got == [2.0, 0.5]                      # every rank sees the maximum
        assert value == pytest.approx(2 * (64 << 20) / 2e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 1.5], 1, "cpu") == [3.0, 1.5]
    assert bench.replica_algbw(1, 1e9, 1000.0) == pytest.approx(1.0)


def test_reference_arm_ranks_other_than_0_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    def no_oracle(*a, **k):
        raise AssertionError("rank 1 must not run the oracle")
    monkeypatch.setattr(bench, "ParallelOracle", no_oracle)
    assert bench.run_reference(None, bench.WORKLOADS["ring_fp32_p8"]) is None


def test_l2_note_names_the_case_that_applies():
    """AllReduce / ReduceScatter inputs (P n b) larger than the 129 MB L2;
    an AllGather whose inputs fit but whose outputs (P n b) do not; and the
    L2-resident latency regime."""
    assert bench.l2_note("allreduce", 8, 64 << 20).startswith("inputs (512 MiB) larger")
    assert bench.l2_note("reducescatter", 32, 32 << 20).startswith("inputs (1024 MiB) larger")
    ag = bench.l2_note("allgather", 8, 64 << 20)
    assert ag.startswith("inputs 64 MiB; every step writes 512 MiB")
    assert bench.l2_note("allreduce", 8, 16 << 10) == "L2-resident (hot-cache latency regime)"
