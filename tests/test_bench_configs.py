"""bench.py times every configuration of the benchmark in its default run:
the Ring fp32 P = 8 64 MiB AllReduce is the headline, and the `configs`
array of the same line holds the rest.  These CPU checks keep that list
complete and consistent (no GPU needed)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sweep():
    return [bench.WORKLOADS[k] for group in bench.SWEEP for k in group]


def test_sweep_names_known_workloads_and_shares_inputs_per_group():
    for group in bench.SWEEP:
        recipes = {(bench.WORKLOADS[k]["dtype"], bench.WORKLOADS[k]["P"], bench.WORKLOADS[k]["n"],
                    bench.WORKLOADS[k]["scale"]) for k in group}
        assert len(recipes) == 1, group  # one input draw per group
    names = [k for g in bench.SWEEP for k in g]
    assert len(names) == len(set(names))
    assert "ring_fp32_p8" not in names  # the headline is the line's own value


def test_sweep_covers_every_large_configuration():
    have = {(w["algo"], w["coll"], w["P"], w["n"], w["dtype"], w["op"], w["mode"], w["p_intra"],
             w["loop_bytes"]) for w in _sweep()}
    want = set()
    # Ring fp32 P=8 64 MiB: ReduceScatter and AllGather alone, and step mode
    for coll in ("reducescatter", "allgather"):
        for mode in ("fused", "step"):
            want.add(("ring", coll, 8, 16777216, "float32", "sum", mode, 1, 0))
    want.add(("ring", "allreduce", 8, 16777216, "float32", "sum", "step", 1, 0))
    # Ring and RHD bf16 P=8 128 MiB, sum and max
    for algo in ("ring", "rhd"):
        for op in ("sum", "max"):
            for mode in ("fused", "step"):
                want.add((algo, "allreduce", 8, 67108864, "bfloat16", op, mode, 1, 0))
    # Pipeline 4 x 8 fp32 32 MiB: AllReduce / ReduceScatter / AllGather, the
    # step mode with the 64 MiB loop limit; the plain hierarchical AllReduce
    for coll in ("allreduce", "reducescatter", "allgather"):
        want.add(("pipeline", coll, 32, 8388608, "float32", "sum", "fused", 8, 0))
        want.add(("pipeline", coll, 32, 8388608, "float32", "sum", "step", 8, 64 << 20))
    for mode in ("fused", "step"):
        want.add(("hier", "allreduce", 32, 8388608, "float32", "sum", mode, 8, 0))
    assert want <= have, sorted(want - have)


def test_headline_is_the_ring_fp32_allreduce():
    w = bench.WORKLOADS["ring_fp32_p8"]
    assert (w["algo"], w["coll"], w["P"], w["n"], w["dtype"], w["mode"]) == \
        ("ring", "allreduce", 8, 16777216, "float32", "fused")
