"""Pins of the CPU oracle against what the pages and mathematics fix.

These tests never touch the GPU or the product library.  Each pin is chosen
so that a plausible slip in the oracle (a dropped or doubled contribution, a
wrong partner or segment index, a swapped copy/reduce, a wrong rounding
constant, a wrong loop slice) fails at least one of them:

* the definition Y[j] = (+)_i X_i[j] (int32 exact with wrap; max/min exact),
  evaluated here with numpy, not with the oracle;
* every output element carries every rank exactly once (symbolic replay);
* the association trees equal the closed forms of each schedule, and the
  numeric replay equals numpy / torch evaluating those closed forms;
* the worked examples, step counts and traffic figures the pages print
  (tests/golden/), and the Table 1 closed forms of the RHD article;
* partner symmetry, race freedom inside a step, loop invariance;
* the bf16 rounding against torch and against exact rational rounding;
* the fp64 direct reference against numpy and the error bound.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import hc_inputs
import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ALGOS = ("ring", "rhd", "pipeline")
COLLS = ("allreduce", "reducescatter", "allgather")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def pipeline_intra(P):
    """A non-trivial ranks-per-server for P (largest proper divisor <= 8)."""
    for d in (8, 4, 3, 2):
        if P % d == 0 and P // d >= 2:
            return d
    return 1


def pick_intra(algo, P):
    return pipeline_intra(P) if algo == "pipeline" else 1


# ---------------------------------------------------------------------------
# closed-form trees (built from the pages' descriptions, independently of the
# oracle's step machinery)
# ---------------------------------------------------------------------------
def chain(leaves):
    t = leaves[0]
    for x in leaves[1:]:
        t = (t, x)
    return t


def balanced(leaves):
    if len(leaves) == 1:
        return leaves[0]
    h = len(leaves) // 2
    return (balanced(leaves[:h]), balanced(leaves[h:]))


def ring_tree(P, k):
    """Segment k starts at rank k+1 and ends at its owner k."""
    return chain([(k + 1 + i) % P for i in range(P)])


def rhd_tree(P):
    """Fold pairs (2i, 2i+1), i < r, then pairwise combination over the
    power-of-two core, lowest partner bit first."""
    pp = 1 << (P.bit_length() - 1)
    r = P - pp
    u = [(2 * v, 2 * v + 1) if v < r else v + r for v in range(pp)]
    return balanced(u)


def pipe_tree(P, p_intra, k):
    p_inter = P // p_intra
    s, l = divmod(k, p_intra)
    parts = []
    for i in range(1, p_inter + 1):
        sp = (s + i) % p_inter
        parts.append(chain([sp * p_intra + (l + j) % p_intra for j in range(p_intra)]))
    return chain(parts)


def expected_tree(algo, coll, P, p_intra, k):
    if algo == "ring":
        return ring_tree(P, k)
    if algo == "rhd":
        return rhd_tree(P)
    return pipe_tree(P, p_intra, k)


def parse_expr(s):
    pos = 0

    def rec():
        nonlocal pos
        if s[pos] == "(":
            pos += 1
            a = rec()
            assert s[pos] == "+"
            pos += 1
            b = rec()
            assert s[pos] == ")"
            pos += 1
            return (a, b)
        if s[pos] == "?":
            pos += 1
            return "?"
        assert s[pos] == "X"
        pos += 1
        j = pos
        while pos < len(s) and s[pos].isdigit():
            pos += 1
        return int(s[j:pos])

    t = rec()
    assert pos == len(s)
    return t


def canon(t):
    """Order-free form: the two operands of every (+) sorted (the four ops are
    commutative bit for bit, so only the pairing matters)."""
    if isinstance(t, tuple):
        a, b = canon(t[0]), canon(t[1])
        return (a, b) if repr(a) <= repr(b) else (b, a)
    return t


def eval_tree(t, leaf, op):
    if isinstance(t, tuple):
        return op(eval_tree(t[0], leaf, op), eval_tree(t[1], leaf, op))
    return leaf(t)


def owner_rows(coll, P, segs):
    """(rank, segment) pairs whose value is the collective's result."""
    if coll == "reducescatter":
        return [(r, r) for r in range(P)]
    return [(r, k) for r in range(P) for k in range(len(segs))]


# ---------------------------------------------------------------------------
# layout and slicer
# ---------------------------------------------------------------------------
def test_layout_small_cases():
    # n=10 fp32 over 4 segments: ceil(10/4)=3 -> rounded to 4 elements (16 B)
    assert O.segments("ring", "allreduce", 4, 10, "float32") == [(0, 4), (4, 4), (8, 2), (10, 0)]
    # bf16 rounds to 8 elements
    assert O.segments("ring", "allreduce", 3, 20, "bfloat16") == [(0, 8), (8, 8), (16, 4)]
    # RHD AllReduce uses p' = 4 segments for P = 5
    assert O.num_segments("rhd", "allreduce", 5) == 4
    assert O.num_segments("rhd", "reducescatter", 5) == 5
    assert O.segments("ring", "allreduce", 4, 0, "float32") == [(0, 0)] * 4


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", COLLS)
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_layout_tiles_and_aligns(algo, coll, dtype):
    A = 16 // O.ESIZE[dtype]
    for P in (1, 2, 3, 5, 8, 12, 32, 64):
        for n in (0, 1, 7, 64, 1000, 4099):
            segs = O.segments(algo, coll, P, n, dtype)
            pos = 0
            for off, ln in segs:
                assert off == pos and ln >= 0
                assert off % A == 0 or off == n
                pos += ln
            assert pos == n
            lens = [ln for _, ln in segs]
            # every segment but trailing ones has the same length
            full = [ln for ln in lens if ln == lens[0]]
            assert lens[:len(full)] == full


def test_slicer_pipeline_cfg():
    # 4 servers x 8 ranks, 8,388,608 fp32 per rank, 64 MiB per loop
    c, loops, tail = O.slicer("pipeline", "allreduce", 32, 8388608, "float32", 64 << 20, p_intra=8)
    assert (c, loops, tail) == (74880, 4, 37504)
    assert c % 32 == 0                       # 128-byte granule
    assert O.slicer("ring", "allreduce", 8, 1 << 20, "float32", 0) == (131072, 1, 131072)


@pytest.mark.parametrize("algo", ALGOS)
def test_slicer_covers_segments(algo):
    P = 12
    pin = pick_intra(algo, P)
    for n in (1000, 4096, 77777):
        for lb in (4096, 65536, 1 << 20):
            msgs, spl, loops = O.schedule(algo, "allreduce", P, n, "float32", lb, p_intra=pin)
            c, nl, tail = O.slicer(algo, "allreduce", P, n, "float32", lb, p_intra=pin)
            assert nl == loops
            segs = O.segments(algo, "allreduce", P, n, "float32")
            for k, (off, ln) in enumerate(segs):
                m = msgs[msgs["seg"] == k]
                for i in range(loops):
                    mi = m[m["loop"] == i]
                    lo, hi = off + i * c, min(off + (i + 1) * c, off + ln)
                    if lo >= hi:
                        assert mi.size == 0
                    else:
                        assert np.all(mi["lo"] == lo) and np.all(mi["hi"] == hi)


# ---------------------------------------------------------------------------
# definition
# ---------------------------------------------------------------------------
def np_definition(X, op, dtype):
    if dtype == "int32":
        x = X.astype(np.int64)
        if op == "sum":
            return (x.sum(0) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)
        if op == "prod":
            acc = np.ones(X.shape[1], dtype=np.uint64)
            for row in X.astype(np.int64):
                acc = (acc * (row.astype(np.uint64) & np.uint64(0xFFFFFFFF))) & np.uint64(0xFFFFFFFF)
            return acc.astype(np.uint32).view(np.int32)
        return X.max(0) if op == "max" else X.min(0)
    if dtype == "float32":
        return X.max(0) if op == "max" else X.min(0)
    import torch
    t = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16)
    r = t.max(0).values if op == "max" else t.min(0).values
    return r.view(torch.int16).numpy().view(np.uint16)


def collective_result(coll, Y, X, algo, P, n, dtype, ref):
    """Check a replay Y against a per-element reference `ref` (length n)."""
    segs = O.segments(algo, coll, P, n, dtype)
    if coll == "allreduce":
        for r in range(P):
            np.testing.assert_array_equal(Y[r], ref)
    elif coll == "reducescatter":
        for r in range(P):
            off, ln = segs[r]
            np.testing.assert_array_equal(Y[r, off:off + ln], ref[off:off + ln])
    else:
        gathered = np.empty_like(X[0])
        for k, (off, ln) in enumerate(segs):
            gathered[off:off + ln] = X[k, off:off + ln]
        for r in range(P):
            np.testing.assert_array_equal(Y[r], gathered)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", COLLS)
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_definition_int32(algo, coll, op):
    for P in (1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16):
        pin = pick_intra(algo, P)
        for n in (1, 13, 100):
            X = hc_inputs.uniform_int32(P, n, seed=P * 1000 + n)
            if op == "prod":
                X = (X % 7).astype(np.int32)
            Y = O.replay(algo, coll, X, op, "int32", p_intra=pin)
            collective_result(coll, Y, X, algo, P, n, "int32", np_definition(X, op, "int32"))


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", ["allreduce", "reducescatter"])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("op", ["max", "min"])
def test_definition_float_maxmin(algo, coll, dtype, op):
    for P in (2, 3, 5, 8, 12):
        pin = pick_intra(algo, P)
        X = hc_inputs.rank_buffers(dtype, P, 77, seed=P, scale=1.0)
        Y = O.replay(algo, coll, X, op, dtype, p_intra=pin)
        collective_result(coll, Y, X, algo, P, 77, dtype, np_definition(X, op, dtype))


def test_cfg_int32_ring4_rhd5():
    """int32 sum, values uniform in [-1000, 1000] from seed 0: Ring over ranks
    0..3 and RHD over all 5 rows give the exact sum on every rank."""
    X = hc_inputs.uniform_int32(5, 4096, seed=0)
    Y = O.replay("ring", "allreduce", X[:4].copy(), "sum", "int32")
    assert np.array_equal(Y, np.broadcast_to(X[:4].astype(np.int64).sum(0), Y.shape))
    Y = O.replay("rhd", "allreduce", X, "sum", "int32")
    assert np.array_equal(Y, np.broadcast_to(X.astype(np.int64).sum(0), Y.shape))


# ---------------------------------------------------------------------------
# every rank contributes exactly once; trees equal the closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", COLLS)
def test_each_rank_exactly_once(algo, coll):
    Ps = list(range(1, 34)) + [40, 48, 63, 64]
    for P in Ps:
        pin = pick_intra(algo, P)
        S = O.num_segments(algo, coll, P)
        n = 4 * S + 3  # ragged: the last segment is short
        O.sym_reset()
        Y = O.replay_sym(algo, coll, P, n, p_intra=pin)
        segs = O.segments(algo, coll, P, n, "float32")
        for r, k in owner_rows(coll, P, segs):
            off, ln = segs[k]
            for j in (off, off + ln - 1):
                if ln == 0:
                    continue
                cnt = O.sym_leaves(Y[r, j])
                if coll == "allgather":
                    expect = np.zeros_like(cnt)
                    expect[k] = 1
                else:
                    expect = np.zeros_like(cnt)
                    expect[:P] = 1
                assert np.array_equal(cnt, expect), (P, r, k, O.sym_string(Y[r, j]))


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", ["allreduce", "reducescatter"])
def test_trees_equal_closed_forms(algo, coll):
    for P in (1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 24, 32):
        pin = pick_intra(algo, P)
        S = O.num_segments(algo, coll, P)
        n = 4 * S
        O.sym_reset()
        Y = O.replay_sym(algo, coll, P, n, p_intra=pin)
        segs = O.segments(algo, coll, P, n, "float32")
        for r, k in owner_rows(coll, P, segs):
            off, _ = segs[k]
            got = canon(parse_expr(O.sym_string(Y[r, off])))
            if algo == "rhd" and coll == "reducescatter":
                want = canon(rhd_tree(P))
            else:
                want = canon(expected_tree(algo, coll, P, pin, k))
            assert got == want, (algo, coll, P, r, k)


def test_rhd_five_rank_tree_literal():
    """((X0+X1)+X2)+(X3+X4): fold rank1 into rank0, then the 4-rank core
    pairs {0,2} and {3,4} first, lowest partner bit first."""
    O.sym_reset()
    Y = O.replay_sym("rhd", "allreduce", 5, 16)
    want = canon(parse_expr("(((X0+X1)+X2)+(X3+X4))"))
    for r in range(5):
        for j in range(16):
            assert canon(parse_expr(O.sym_string(Y[r, j]))) == want


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", ["allreduce", "reducescatter"])
def test_fp32_replay_equals_closed_form_in_numpy(algo, coll):
    """Numeric replay (binary32 per step) == numpy float32 evaluating the
    closed-form tree, bit for bit; catches a wrong association anywhere."""
    for P in (2, 3, 5, 8, 12, 16):
        pin = pick_intra(algo, P)
        n = 8 * O.num_segments(algo, coll, P) + 5
        # tree-discriminating data: mixes magnitudes so that any re-association
        # changes low bits
        rng = np.random.default_rng(P)
        X = (rng.standard_normal((P, n)) * np.exp2(rng.integers(-12, 12, (P, n)))).astype(np.float32)
        Y = O.replay(algo, coll, X, "sum", "float32", p_intra=pin)
        segs = O.segments(algo, coll, P, n, "float32")
        for r, k in owner_rows(coll, P, segs):
            off, ln = segs[k]
            if ln == 0:
                continue
            t = rhd_tree(P) if algo == "rhd" else expected_tree(algo, coll, P, pin, k)
            want = eval_tree(t, lambda i: X[i, off:off + ln], lambda a, b: a + b)
            np.testing.assert_array_equal(Y[r, off:off + ln].view(np.uint32),
                                          np.asarray(want, dtype=np.float32).view(np.uint32))


@pytest.mark.parametrize("algo", ALGOS)
def test_bf16_replay_equals_closed_form_in_torch(algo):
    """bf16 per-step rounding == torch bfloat16 arithmetic on the closed-form
    tree (torch computes a bf16 add/mul in binary32 and rounds to nearest even)."""
    import torch
    for P, op in ((3, "sum"), (5, "sum"), (8, "sum"), (12, "sum"), (8, "prod")):
        pin = pick_intra(algo, P)
        n = 16 * O.num_segments(algo, "allreduce", P) + 9
        X = hc_inputs.gradients_bf16(P, n, seed=P, scale=1.0)
        Y = O.replay(algo, "allreduce", X, op, "bfloat16", p_intra=pin)
        T = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16)
        segs = O.segments(algo, "allreduce", P, n, "bfloat16")
        f = (lambda a, b: a + b) if op == "sum" else (lambda a, b: a * b)
        for k, (off, ln) in enumerate(segs):
            if ln == 0:
                continue
            t = rhd_tree(P) if algo == "rhd" else expected_tree(algo, "allreduce", P, pin, k)
            want = eval_tree(t, lambda i: T[i, off:off + ln], f)
            want = want.view(torch.int16).numpy().view(np.uint16)
            for r in range(P):
                np.testing.assert_array_equal(Y[r, off:off + ln], want)


def test_int32_prod_and_sum_wrap():
    X = np.array([[2**30, 3], [4, 2**31 - 1], [5, 2]], dtype=np.int32)
    for algo in ALGOS:
        Y = O.replay(algo, "allreduce", X, "sum", "int32", p_intra=1 if algo != "pipeline" else 3)
        want = ((X.astype(np.int64).sum(0) + 2**31) % 2**32 - 2**31).astype(np.int32)
        assert np.array_equal(Y[0], want)
        Y = O.replay(algo, "allreduce", X, "prod", "int32", p_intra=1 if algo != "pipeline" else 3)
        want = [(2**30 * 4 * 5) % 2**32, (3 * (2**31 - 1) * 2) % 2**32]
        want = np.array([(w + 2**31) % 2**32 - 2**31 for w in want], dtype=np.int32)
        assert np.array_equal(Y[0], want)


def test_totalorder_special_values():
    """max/min follow IEEE 754 totalOrder: -0 < +0, -NaN < -inf, +inf < +NaN."""
    pz, nz = np.float32(0.0), np.float32(-0.0)
    qnan = np.array([0x7FC00000], dtype=np.uint32).view(np.float32)[0]
    nnan = np.array([0xFFC00000], dtype=np.uint32).view(np.float32)[0]
    inf = np.float32(np.inf)
    cases = [  # (a, b, max, min) as float32
        (pz, nz, pz, nz),
        (nz, pz, pz, nz),
        (qnan, inf, qnan, inf),
        (nnan, -inf, -inf, nnan),
        (np.float32(1), qnan, qnan, np.float32(1)),
    ]
    for a, b, mx, mn in cases:
        X = np.array([[a], [b]], dtype=np.float32)
        for op, want in (("max", mx), ("min", mn)):
            for algo in ("ring", "rhd"):
                Y = O.replay(algo, "allreduce", X, op, "float32")
                assert Y.view(np.uint32)[0, 0] == np.float32(want).view(np.uint32)
                assert Y.view(np.uint32)[1, 0] == np.float32(want).view(np.uint32)
            raw, _, _ = O.direct(X, op, "float32")
            assert raw.view(np.uint32)[0] == np.float32(want).view(np.uint32)
    # bf16: +0 = 0x0000, -0 = 0x8000
    X = np.array([[0x8000], [0x0000]], dtype=np.uint16)
    assert O.replay("ring", "allreduce", X, "max", "bfloat16")[0, 0] == 0x0000
    assert O.replay("ring", "allreduce", X, "min", "bfloat16")[0, 0] == 0x8000


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
def test_bf16_rounding_matches_torch():
    import torch
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    special = np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, -3.4e38,
                        1e-40, -1e-40, 1.5e-45], dtype=np.float32)
    f = np.concatenate([f, special])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.f32_to_bf16(float(x)) for x in f], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


def _bf16_value(h):
    return Fraction(float(np.array([int(h) << 16], dtype=np.uint32).view(np.float32)[0]))


def _exact_rne_bf16(x: Fraction):
    """Round an exact rational to the nearest bf16 (ties to even mantissa) by
    comparing exact distances to the bracketing bf16 values."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    ax = -x if x < 0 else x
    # find the largest finite bf16 magnitude <= ax by bisection over bit patterns
    lo, hi = 0, 0x7F7F
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if _bf16_value(mid) <= ax:
            lo = mid
        else:
            hi = mid - 1
    below = lo
    above = below + 1
    db = ax - _bf16_value(below)
    da = _bf16_value(above) - ax if above <= 0x7F7F else None
    if da is None:
        # beyond the largest finite value: ties and overflow round as IEEE
        half_ulp = (_bf16_value(0x7F7F) - _bf16_value(0x7F7E)) / 2
        pick = below if db < half_ulp else 0x7F80
    elif db < da:
        pick = below
    elif da < db:
        pick = above
    else:
        pick = below if below % 2 == 0 else above
    return sign | pick


def test_bf16_step_rounding_is_single_rounding_of_exact():
    """Rounding fp32(a) (+) fp32(b) to bf16 gives the bf16 nearest the exact
    a (+) b, for add and mul (the reading of 'bf16 rounded after each step')."""
    rng = np.random.default_rng(11)
    n = 3000
    exps = rng.integers(-20, 20, size=(2, n))
    mant = rng.integers(0, 128, size=(2, n))
    sgn = rng.integers(0, 2, size=(2, n))
    H = ((sgn << 15) | ((exps + 127) << 7) | mant).astype(np.uint16)
    for op in ("sum", "prod"):
        Y = O.replay("ring", "allreduce", H.T.copy().reshape(n, 2).T.copy(), op, "bfloat16")
        for j in range(n):
            a, b = _bf16_value(H[0, j]), _bf16_value(H[1, j])
            exact = a + b if op == "sum" else a * b
            want = _exact_rne_bf16(exact)
            got = int(Y[0, j])
            if exact == 0:
                assert got & 0x7FFF == 0
            else:
                assert got == want, (op, hex(H[0, j]), hex(H[1, j]), hex(got), hex(want))


# ---------------------------------------------------------------------------
# direct reference and error bound
# ---------------------------------------------------------------------------
def test_direct_matches_numpy():
    X = hc_inputs.gradients_f32(7, 5000, seed=3, scale=1.0)
    _, y64, s1 = O.direct(X, "sum", "float32")
    np.testing.assert_allclose(y64, X.astype(np.float64).sum(0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(s1, np.abs(X.astype(np.float64)).sum(0), rtol=1e-15)
    _, p64, _ = O.direct(X, "prod", "float32")
    np.testing.assert_allclose(p64, X.astype(np.float64).prod(0), rtol=1e-13)
    Xi = hc_inputs.uniform_int32(7, 5000, seed=3)
    raw, y64, _ = O.direct(Xi, "sum", "int32")
    assert np.array_equal(raw, Xi.astype(np.int64).sum(0).astype(np.int32))
    assert np.array_equal(y64, Xi.astype(np.int64).sum(0).astype(np.float64))


def rounding_depth(algo, P, p_intra):
    if algo == "ring":
        return P - 1
    if algo == "rhd":
        pp = 1 << (P.bit_length() - 1)
        return int(math.log2(pp)) + (1 if P > pp else 0)
    return (p_intra - 1) + (P // p_intra - 1)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_error_bound_vs_fp64(algo, dtype):
    """|y - y64| <= g_d * sum|x| per element (g_d = d u / (1 - d u), d roundings
    on the element's path), and the normwise tolerance 1e-5 (fp32) / 1e-2 (bf16)."""
    u = 2.0 ** -24 if dtype == "float32" else 2.0 ** -8
    for P in (4, 5, 8, 12):
        pin = pick_intra(algo, P)
        n = 20000
        X = hc_inputs.rank_buffers(dtype, P, n, seed=P)
        Y = O.replay(algo, "allreduce", X, "sum", dtype, p_intra=pin)
        _, y64, s1 = O.direct(X, "sum", dtype)
        if dtype == "float32":
            y = Y[0].astype(np.float64)
        else:
            y = (Y[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        d = rounding_depth(algo, P, pin)
        gam = d * u / (1 - d * u)
        assert np.all(np.abs(y - y64) <= gam * s1 + 1e-300)
        rel = np.linalg.norm(y - y64) / np.linalg.norm(y64)
        assert rel <= (1e-5 if dtype == "float32" else 1e-2)


# ---------------------------------------------------------------------------
# schedules: printed examples, step counts, traffic, symmetry, races, loops
# ---------------------------------------------------------------------------
def steps_of(msgs, loop=0):
    m = msgs[msgs["loop"] == loop]
    return [m[m["step"] == s] for s in range(int(m["step"].max()) + 1)] if m.size else []


def test_rhd_five_rank_worked_example():
    g = {row[0]: row[1:] for row in read_golden("rhd_5rank_allreduce.txt")}
    P = int(g["ranks"][0])
    n = 4 * 64
    msgs, spl, _ = O.schedule("rhd", "allreduce", P, n)
    assert spl == int(g["steps"][0])
    st = steps_of(msgs)
    kinds = {"reduce": O.REDUCE, "copy": O.COPY}
    first, last = st[0], st[-1]
    assert set(first["src"]) == {int(g["fold_src"][0])} and set(first["dst"]) == {int(g["fold_dst"][0])}
    assert set(first["kind"]) == {kinds[g["fold_kind"][0]]}
    assert (first["hi"] - first["lo"]).sum() == n
    assert set(last["src"]) == {int(g["unfold_src"][0])} and set(last["dst"]) == {int(g["unfold_dst"][0])}
    assert set(last["kind"]) == {kinds[g["unfold_kind"][0]]}
    assert (last["hi"] - last["lo"]).sum() == n
    core = set(int(x) for x in g["core_ranks"])
    nh, nd = int(g["core_halving_rounds"][0]), int(g["core_doubling_rounds"][0])
    middle = st[1:-1]
    assert len(middle) == nh + nd
    for i, s in enumerate(middle):
        assert set(s["src"]) | set(s["dst"]) <= core
        assert set(s["kind"]) == {O.REDUCE if i < nh else O.COPY}
        # each core rank sends to exactly one partner, and partners are mutual
        pairs = set(zip(s["src"].tolist(), s["dst"].tolist()))
        partner = dict(pairs)
        assert len(partner) == len(core) and all(partner[partner[a]] == a for a in partner)
        # halving: n/2 then n/4 per rank; doubling mirrors it
        per_rank = {a: int((s["hi"] - s["lo"])[s["src"] == a].sum()) for a in core}
        expect = n >> (i + 1) if i < nh else n >> (nh + nd - i)
        assert set(per_rank.values()) == {expect}


def test_printed_step_counts():
    for algo, coll, P, steps in read_golden("step_counts.txt"):
        P, steps = int(P), int(steps)
        _, spl, _ = O.schedule(algo, coll, P, 16 * P)
        assert spl == steps, (algo, coll, P)


@pytest.mark.parametrize("P", list(range(1, 70)))
def test_step_count_closed_forms(P):
    """Ring 2(P-1); RHD AllReduce 2 log2 P (power of two) or 2 floor(log P) + 2
    = 2 ceil(log2 P); RHD ReduceScatter / AllGather log2 P or floor(log P) + 2
    (Table 1 of the RHD article)."""
    n = 16 * P
    fl = P.bit_length() - 1
    pow2 = (P & (P - 1)) == 0
    assert O.schedule("ring", "allreduce", P, n)[1] == 2 * (P - 1)
    assert O.schedule("ring", "reducescatter", P, n)[1] == P - 1
    assert O.schedule("ring", "allgather", P, n)[1] == P - 1
    ar = O.schedule("rhd", "allreduce", P, n)[1]
    assert ar == (2 * fl if pow2 else 2 * fl + 2)
    if P > 1:
        assert ar == 2 * math.ceil(math.log2(P))
    for coll in ("reducescatter", "allgather"):
        assert O.schedule("rhd", coll, P, n)[1] == (fl if pow2 else fl + 2)


@pytest.mark.parametrize("p_inter,p_intra", [(4, 8), (3, 2), (2, 4), (1, 4), (4, 1), (5, 3)])
def test_pipeline_step_structure(p_inter, p_intra):
    """Table 1 of the Pipeline article: (p_inter - 1) overlapped steps plus one
    intra-server step per phase; AllReduce twice that; one block per link per
    step (s/p in the table)."""
    P = p_inter * p_intra
    n = 64 * P
    L = n // P
    per_phase = (p_inter - 1) + (1 if p_intra > 1 else 0)
    assert O.schedule("pipeline", "allgather", P, n, p_intra=p_intra)[1] == per_phase
    assert O.schedule("pipeline", "reducescatter", P, n, p_intra=p_intra)[1] == per_phase
    msgs, spl, _ = O.schedule("pipeline", "allreduce", P, n, p_intra=p_intra)
    assert spl == 2 * per_phase
    assert np.all(msgs["hi"] - msgs["lo"] == L)
    for s in steps_of(msgs):
        links = list(zip(s["src"].tolist(), s["dst"].tolist()))
        assert len(links) == len(set(links))      # one block per link per step
        for a, b in links:
            sa, sb = divmod(a, p_intra), divmod(b, p_intra)
            inter = sa[0] != sb[0]
            if inter:    # inter-server links join equal local indices, ring s -> s+1
                assert sa[1] == sb[1] and sb[0] == (sa[0] + 1) % p_inter
    # AllGather: in the overlapped steps a rank forwards one block on the ring
    # and the same block inside its server
    ag, _, _ = O.schedule("pipeline", "allgather", P, n, p_intra=p_intra)
    for s in steps_of(ag):
        for a in range(P):
            sent = s[s["src"] == a]
            assert len(set(sent["seg"].tolist())) <= 1


def test_pipeline_allgather_narrative():
    rows = read_golden("pipeline_allgather_narrative.txt")
    P = int(rows[0][1])
    pin = int(rows[1][1])
    msgs, _, _ = O.schedule("pipeline", "allgather", P, 16 * P, p_intra=pin)
    st = steps_of(msgs)
    for step, kind, src, dst, owner in rows[2:]:
        s = st[int(step) - 1]
        hit = s[(s["src"] == int(src)) & (s["dst"] == int(dst)) & (s["seg"] == int(owner))]
        assert hit.size == 1, (step, src, dst)
        inter = int(src) // pin != int(dst) // pin
        assert inter == (kind == "inter")


def bytes_sent(msgs, P):
    out = np.zeros(P, dtype=np.int64)
    np.add.at(out, msgs["src"], msgs["hi"] - msgs["lo"])
    return out


def test_printed_traffic():
    for algo, coll, P, factor in read_golden("traffic.txt"):
        P, factor = int(P), float(factor)
        n = 64 * P
        msgs, _, _ = O.schedule(algo, coll, P, n)
        assert np.all(bytes_sent(msgs, P) == factor * n)


@pytest.mark.parametrize("P", [2, 3, 4, 5, 6, 7, 8, 12, 16, 31, 32, 64])
def test_traffic_closed_forms(P):
    n = 16 * P * 8  # divisible so that all blocks are equal
    sent = bytes_sent(O.schedule("ring", "allreduce", P, n)[0], P)
    assert np.all(sent == 2 * (P - 1) * n // P)
    sent = bytes_sent(O.schedule("ring", "reducescatter", P, n)[0], P)
    assert np.all(sent == (P - 1) * n // P)
    if P & (P - 1) == 0:
        sent = bytes_sent(O.schedule("rhd", "reducescatter", P, n)[0], P)
        assert np.all(sent == (P - 1) * n // P)
        sent = bytes_sent(O.schedule("rhd", "allreduce", P, n)[0], P)
        assert np.all(sent == 2 * (P - 1) * n // P)


def per_step_max(msgs, P):
    out = []
    for s in steps_of(msgs):
        out.append(int(bytes_sent(s, P).max()))
    return out


@pytest.mark.parametrize("P", list(range(3, 65)))
def test_rhd_table1_exchange_sizes(P):
    """RHD article Table 1: non-power-of-two ReduceScatter = Reduce (n) + k
    rounds whose largest exchange is ceil(p / 2^i) n / p, i = 1..k (the
    multiset the table lists) + Scatter (n / p), with its lower and upper
    bounds; AllGather the same; AllReduce critical path
    (2 (p' - 1) / p' + 2) n."""
    if P & (P - 1) == 0:
        return
    n = P * 16 * 4
    blk = n // P
    k = P.bit_length() - 1
    for coll in ("reducescatter", "allgather"):
        mx = per_step_max(O.schedule("rhd", coll, P, n)[0], P)
        assert len(mx) == k + 2
        ends = sorted([mx[0], mx[-1]])
        assert ends == [blk, n] or ends == [blk, blk]
        rounds = mx[1:-1]
        assert sorted(rounds) == sorted(math.ceil(P / 2 ** i) * blk for i in range(1, k + 1))
        total = sum(rounds)
        assert (k + 2 ** k - 1) * blk <= total <= (2 ** (k + 1) - 2) * blk
    rs = per_step_max(O.schedule("rhd", "reducescatter", P, n)[0], P)
    assert rs[0] == n and rs[-1] == blk
    pp = 1 << k
    n_ar = pp * 64  # p' equal blocks of a multiple of 16 bytes
    mx = per_step_max(O.schedule("rhd", "allreduce", P, n_ar)[0], P)
    assert Fraction(sum(mx), n_ar) == 2 * Fraction(pp - 1, pp) + 2


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", COLLS)
def test_partners_and_no_intra_step_races(algo, coll):
    """In every step: RHD partners are mutual and unique, Ring ranks send to
    q+1 only; and no element written in a step is read in that step by
    another message, so every step can run in place."""
    for P in (2, 3, 4, 5, 6, 8, 9, 12, 16):
        pin = pick_intra(algo, P)
        n = 16 * P + 4
        msgs, _, _ = O.schedule(algo, coll, P, n, p_intra=pin)
        for s in steps_of(msgs):
            if algo == "ring":
                assert np.all(s["dst"] == (s["src"] + 1) % P)
            if algo == "rhd":
                pairs = set(zip(s["src"].tolist(), s["dst"].tolist()))
                srcs = [a for a, _ in pairs]
                assert len(srcs) == len(set(srcs))
                if len(set(s["kind"])) == 1 and len(pairs) > 1 and pairs != {(a, b) for a, b in pairs if a > b}:
                    pass
            writes = {}
            for m in s:
                writes.setdefault(int(m["dst"]), []).append((int(m["lo"]), int(m["hi"])))
            for m in s:
                for lo, hi in writes.get(int(m["src"]), []):
                    assert hi <= m["lo"] or m["hi"] <= lo, (algo, coll, P)


def test_rhd_partners_mutual_in_core_rounds():
    for P in range(2, 65):
        pp = 1 << (P.bit_length() - 1)
        r = P - pp
        msgs, _, _ = O.schedule("rhd", "allreduce", P, 64 * pp)  # no empty blocks
        st = steps_of(msgs)
        core = st[1:-1] if r else st
        for s in core:
            partner = {}
            for a, b in zip(s["src"].tolist(), s["dst"].tolist()):
                assert partner.setdefault(a, b) == b
            assert all(partner[b] == a for a, b in partner.items())
            assert len(partner) == pp


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("coll", COLLS)
def test_loops_do_not_change_results(algo, coll):
    P = 12
    pin = pick_intra(algo, P)
    n = 50003
    X = hc_inputs.gradients_f32(P, n, seed=7, scale=1.0)
    Y0 = O.replay(algo, coll, X, "sum", "float32", p_intra=pin)
    for lb in (8192, 100000):
        assert O.slicer(algo, coll, P, n, "float32", lb, p_intra=pin)[1] > 1
        Y1 = O.replay(algo, coll, X, "sum", "float32", loop_bytes=lb, p_intra=pin)
        np.testing.assert_array_equal(Y0.view(np.uint32), Y1.view(np.uint32))


def test_sampled_replay_equals_full_replay():
    P, n = 8, 4099
    X = hc_inputs.gradients_f32(P, n, seed=9)
    J = hc_inputs.sample_indices(n, 300, seed=2)
    for algo in ALGOS:
        pin = pick_intra(algo, P)
        full = O.replay(algo, "allreduce", X, "sum", "float32", p_intra=pin)
        part = O.replay(algo, "allreduce", X, "sum", "float32", p_intra=pin, J=J)
        np.testing.assert_array_equal(full[:, J].view(np.uint32), part.view(np.uint32))


def test_bad_arguments_rejected():
    X = np.zeros((6, 10), dtype=np.float32)
    with pytest.raises(ValueError):
        O.replay("pipeline", "allreduce", X, "sum", "float32", p_intra=4)
    with pytest.raises(ValueError):
        O.replay("ring", "allreduce", X, "sum", "float32", J=np.array([3, 2]))
    with pytest.raises(ValueError):
        O.schedule("ring", "allreduce", 0, 10)


# ---------------------------------------------------------------------------
# RHD Broadcast (Table 1 of the RHD article, Broadcast row)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("P", list(range(1, 41)) + [63, 64])
def test_broadcast_every_rank_gets_the_root_exactly(P):
    n = 20
    for root in range(P):
        O.sym_reset()
        Y = O.replay_sym("rhd", "broadcast", P, n, root=root)
        for r in range(P):
            cnt = O.sym_leaves(Y[r, 0])
            want = np.zeros_like(cnt)
            want[root] = 1
            assert np.array_equal(cnt, want), (P, root, r)
        X = hc_inputs.uniform_int32(P, n, seed=P * 100 + root)
        Yn = O.replay("rhd", "broadcast", X, "sum", "int32", root=root)
        assert np.all(Yn == X[root][None, :])


@pytest.mark.parametrize("P", list(range(1, 65)))
def test_broadcast_schedule_table1(P):
    """ceil(log2 P) steps of n elements each (the row's ceil(log p)(a + n b));
    every non-root rank receives exactly once, the root never; the part1 ranks
    of the root's parity join the distance-halving block and each then sends
    once to its pair partner."""
    n = 64
    pp = 1 << (P.bit_length() - 1)
    r = P - pp
    for root in range(P):
        msgs, spl, _ = O.schedule("rhd", "broadcast", P, n, root=root)
        assert spl == (math.ceil(math.log2(P)) if P > 1 else 0)
        assert np.all(msgs["hi"] - msgs["lo"] == n) and np.all(msgs["kind"] == O.COPY)
        recv = np.bincount(msgs["dst"], minlength=P)
        assert recv[root] == 0 and all(recv[q] == 1 for q in range(P) if q != root)
        par = root & 1
        for s in steps_of(msgs):
            srcs, dsts = s["src"].tolist(), s["dst"].tolist()
            assert len(set(srcs)) == len(srcs) and len(set(dsts)) == len(dsts)
        core = msgs[msgs["step"] < spl - (1 if r else 0)]
        for q in set(core["src"].tolist()) | set(core["dst"].tolist()):
            assert q >= 2 * r or q % 2 == par
        if r:
            last = msgs[msgs["step"] == spl - 1]
            assert sorted(zip(last["src"].tolist(), last["dst"].tolist())) == \
                [(2 * i + par, 2 * i + 1 - par) for i in range(r)]


# ---------------------------------------------------------------------------
# plain hierarchical AllReduce: intra-server RS (mesh) -> inter-server RHD AR
# -> intra-server AG (mesh)
# ---------------------------------------------------------------------------
HIER_SHAPES = [(1, 1), (4, 1), (4, 4), (6, 3), (8, 2), (8, 4), (12, 4), (12, 2), (15, 3),
               (20, 4), (24, 8), (32, 8), (40, 8), (64, 8)]


def hier_tree(P, pin, k):
    pout = P // pin
    pp = 1 << (pout.bit_length() - 1)
    r = pout - pp
    l = k // pp
    I = [chain([s * pin + (l + j) % pin for j in range(pin)]) for s in range(pout)]
    u = [(I[2 * v], I[2 * v + 1]) if v < r else I[v + r] for v in range(pp)]
    return balanced(u)


@pytest.mark.parametrize("P,pin", HIER_SHAPES)
def test_hier_definition_contributions_and_trees(P, pin):
    S = O.num_segments("hier", "allreduce", P, pin)
    n = 4 * S + 3
    for op in ("sum", "prod", "max", "min"):
        X = hc_inputs.uniform_int32(P, n, seed=P + pin)
        if op == "prod":
            X = (X % 5).astype(np.int32)
        Y = O.replay("hier", "allreduce", X, op, "int32", p_intra=pin)
        want = np_definition(X, op, "int32")
        assert all(np.array_equal(Y[r], want) for r in range(P))
    O.sym_reset()
    Ys = O.replay_sym("hier", "allreduce", P, n, p_intra=pin)
    segs = O.segments("hier", "allreduce", P, n, "float32", p_intra=pin)
    for k, (off, ln) in enumerate(segs):
        if ln == 0:
            continue
        for r in range(P):
            cnt = O.sym_leaves(Ys[r, off])
            assert np.all(cnt[:P] == 1) and cnt[P:].sum() == 0
        assert canon(parse_expr(O.sym_string(Ys[0, off]))) == canon(hier_tree(P, pin, k))
    rng = np.random.default_rng(P)
    Xf = (rng.standard_normal((P, n)) * np.exp2(rng.integers(-12, 12, (P, n)))).astype(np.float32)
    Yf = O.replay("hier", "allreduce", Xf, "sum", "float32", p_intra=pin)
    for k, (off, ln) in enumerate(segs):
        if ln == 0:
            continue
        want = eval_tree(hier_tree(P, pin, k), lambda i: Xf[i, off:off + ln], lambda a, b: a + b)
        np.testing.assert_array_equal(Yf[0, off:off + ln].view(np.uint32),
                                      np.asarray(want, np.float32).view(np.uint32))


@pytest.mark.parametrize("P,pin", HIER_SHAPES)
def test_hier_steps_and_traffic(P, pin):
    """One intra-server mesh step, then the RHD AllReduce over servers
    (2 ceil(log2 p_inter) steps, Table 1 of the RHD article), then one mesh
    step.  Traffic per rank for a power-of-two server count:
    (p_intra - 1) n / p_intra twice (mesh RS and mesh AG) plus the RHD
    AllReduce of the intra segment, 2 (p_inter - 1) / p_inter n / p_intra."""
    pout = P // pin
    S = O.num_segments("hier", "allreduce", P, pin)
    n = 16 * S
    msgs, spl, _ = O.schedule("hier", "allreduce", P, n, p_intra=pin)
    want_steps = (2 if pin > 1 else 0) + (2 * math.ceil(math.log2(pout)) if pout > 1 else 0)
    assert spl == want_steps
    if pout & (pout - 1) == 0:
        sent = bytes_sent(msgs, P)
        seg = n // pin
        assert np.all(sent == 2 * (pin - 1) * seg + 2 * (pout - 1) * seg // pout)
    # the intra-server steps stay inside a server; the RHD steps join equal
    # local indices of different servers
    for s in steps_of(msgs):
        intra = [a // pin == b // pin for a, b in zip(s["src"].tolist(), s["dst"].tolist())]
        assert all(intra) or not any(intra)
        if not any(intra):
            assert all(a % pin == b % pin for a, b in zip(s["src"].tolist(), s["dst"].tolist()))


def test_hier_rejects_other_collectives():
    with pytest.raises(ValueError):
        O.schedule("hier", "reducescatter", 8, 64, p_intra=4)
    with pytest.raises(ValueError):
        O.schedule("hier", "allreduce", 8, 64, p_intra=3)
