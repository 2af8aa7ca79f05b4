"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with a retyped copy of itself: each check is
a brute-force sum, a closed form, an identity the pages state (AllReduce =
ReduceScatter + AllGather; the looped form equals the monolithic one; the
permute pairs and shard alignment of the Looped CollectiveEinsum), a
partitioned model equal to its unpartitioned form, or a published test vector.
The last group plants plausible mistakes in the oracle (on the CPU) and shows
that a pin catches each.
"""

import os

import numpy as np
import pytest

import oracle
from oracle import collectives, fused, looped

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(20240601)


def small_ints(shape):
    return RNG.integers(-4, 5, size=shape).astype(np.float64)


# --------------------------------------------------------------------------- einsum


@pytest.mark.parametrize("spec,ls,rs", [
    ("mk,kn->mn", (3, 5), (5, 2)),
    ("mk,kn->mn", (1, 7), (7, 4)),
    ("bmk,bkn->bmn", (2, 3, 4), (2, 4, 5)),
])
def test_einsum_matches_bruteforce(spec, ls, rs):
    a, b = RNG.standard_normal(ls), RNG.standard_normal(rs)
    np.testing.assert_allclose(oracle.einsum(spec, a, b), oracle.einsum_bruteforce(spec, a, b), rtol=1e-13, atol=1e-13)


def test_einsum_rejects_other_specs():
    with pytest.raises(ValueError):
        oracle.einsum("km,kn->mn", np.ones((2, 2)), np.ones((2, 2)))


# --------------------------------------------------------------------- collectives


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dim", [0, 1])
def test_allgather_concatenates_in_partition_order(n, dim):
    shape = (2, 3)
    shards = [np.full(shape, float(s)) for s in range(n)]
    full = oracle.allgather(shards, dim)
    assert full.shape[dim] == n * shape[dim]
    blocks = np.split(full, n, axis=dim)
    for s, blk in enumerate(blocks):
        assert np.all(blk == s)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
def test_reduce_scatter_rank_tagged(n):
    # in_q[j] = (q + 1) * 1000 + (shard of j): rank r must receive
    # 1000 * n(n+1)/2 + n * r everywhere, which identifies both the sum and
    # the shard ID.
    per = 5
    locals_ = []
    for q in range(n):
        locals_.append(np.concatenate([np.full(per, (q + 1) * 1000.0 + s) for s in range(n)]))
    outs = oracle.reduce_scatter(locals_, 0)
    for r, o in enumerate(outs):
        assert o.shape == (per,)
        assert np.all(o == 1000.0 * n * (n + 1) / 2 + n * r)


def test_reduce_scatter_rejects_uneven():
    with pytest.raises(ValueError):
        oracle.reduce_scatter([np.ones(5), np.ones(5)], 0)


@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_allreduce_closed_form_and_replication(n):
    outs = oracle.allreduce([np.full((4, 3), r + 1.0) for r in range(n)])
    assert len(outs) == n
    for o in outs:
        assert np.all(o == n * (n + 1) / 2)
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("n,dim", [(2, 0), (4, 1), (8, 0), (3, 1)])
def test_allreduce_equals_reduce_scatter_then_allgather(n, dim):
    locals_ = [RNG.standard_normal((24, 6 * 4)) for _ in range(n)]
    direct = oracle.allreduce(locals_)
    split = oracle.allreduce_split_rs_ag(locals_, dim)
    for a, b in zip(direct, split):
        assert np.array_equal(a, b)  # same rank-order sums: bit-identical


def _golden_pairs():
    pairs = {}
    with open(os.path.join(GOLDEN, "permute_pairs.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            n, s, d = map(int, line.split())
            pairs.setdefault(n, []).append((s, d))
    return pairs


def test_permute_pairs_match_the_page():
    for n, pairs in _golden_pairs().items():
        assert sorted(oracle.permute_pairs(n)) == sorted(pairs)


def test_collective_permute_moves_left():
    out = oracle.collective_permute(["a", "b", "c", "d"], oracle.permute_pairs(4))
    assert out == ["b", "c", "d", "a"]  # rank r receives what rank r+1 sent


# ------------------------------------------------------------- looped schedules


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_looped_allgather_schedule_aligned_at_start(n):
    trace = []
    shards = [small_ints((2, 3)) for _ in range(n)]
    locs = [small_ints((3, 2)) for _ in range(n)]
    looped.looped_allgather_einsum("mk,kn->mn", "lhs", "m", shards, locs, trace)
    held = {(i, r): s for i, r, s in trace}
    for r in range(n):
        assert held[(0, r)] == r  # aligned at the loop start
        # every rank sees every shard exactly once, moving as a left shift
        assert sorted(held[(i, r)] for i in range(n)) == list(range(n))
        for i in range(1, n):
            assert held[(i, r)] == held[(i - 1, (r + 1) % n)]


@pytest.mark.parametrize("n", [2, 3, 4, 8])
def test_looped_reduce_scatter_schedule_aligned_at_end(n):
    trace = []
    lhs = [small_ints((2 * n, 3)) for _ in range(n)]
    rhs = [small_ints((3, 2)) for _ in range(n)]
    looped.looped_einsum_reduce_scatter("mk,kn->mn", lhs, rhs, "m", trace)
    sid = {(i, q): s for i, q, s in trace}
    for q in range(n):
        assert sid[(n - 1, q)] == q  # aligned at the loop end
        assert sid[(0, q)] != q      # the first DynamicSlice index is not the partition ID
    # output shard r collects the partials of ranks r-1, r-2, ..., r (mod n), in that order
    for r in range(n):
        order = [q for i in range(n) for q in range(n) if sid[(i, q)] == r]
        assert order == [(r - 1 - i) % n for i in range(n)]


# --------------------------------------------------- looped == monolithic (exact)

AG_CASES = [
    # spec, looped side, sliced label, looped shard shape (per rank), other operand shape
    ("mk,kn->mn", "lhs", "m", (3, 5), (5, 4)),        # case 1
    ("mk,kn->mn", "lhs", "k", (6, 2), None),          # case 2 (other = [n*2, 4])
    ("mk,kn->mn", "rhs", "k", (2, 4), None),          # case 2, looped operand on the right
    ("mk,kn->mn", "rhs", "n", (5, 3), (4, 5)),        # case 1, mirrored
    ("bmk,bkn->bmn", "lhs", "b", (2, 3, 4), None),    # case 3
]


def _other_shape(case, n):
    spec, side, lab, shp, other = case
    if other is not None:
        return other
    if lab == "k" and side == "lhs":
        return (shp[1] * n, 4)
    if lab == "k" and side == "rhs":
        return (3, shp[0] * n)
    if lab == "b":
        return (shp[0] * n, shp[2], 5)
    raise AssertionError


@pytest.mark.parametrize("case", AG_CASES)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
def test_looped_allgather_einsum_equals_monolithic(case, n):
    spec, side, lab, shp, _ = case
    shards = [small_ints(shp) for _ in range(n)]
    locs = [small_ints(_other_shape(case, n)) for _ in range(n)]
    a = looped.looped_allgather_einsum(spec, side, lab, shards, locs)
    b = looped.allgather_einsum(spec, side, lab, shards, locs)
    for x, y in zip(a, b):
        assert x.shape == y.shape
        assert np.array_equal(x, y)


@pytest.mark.parametrize("out_label", ["m", "n"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
def test_looped_einsum_rs_equals_monolithic(out_label, n):
    lhs = [small_ints((2 * n, 3)) for _ in range(n)]
    rhs = [small_ints((3, 3 * n)) for _ in range(n)]
    a = looped.looped_einsum_reduce_scatter("mk,kn->mn", lhs, rhs, out_label)
    b = looped.einsum_reduce_scatter("mk,kn->mn", lhs, rhs, out_label)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_case2_k_split_sum_is_the_full_product(n):
    # A [M, K] sliced on K; the sum of the K-block products is A @ B (block identity).
    a_full, b_full = RNG.standard_normal((5, 4 * n)), RNG.standard_normal((4 * n, 3))
    shards = np.split(a_full, n, axis=1)
    out = looped.looped_allgather_einsum("mk,kn->mn", "lhs", "k", shards, [b_full] * n)
    for o in out:
        np.testing.assert_allclose(o, oracle.einsum_bruteforce("mk,kn->mn", a_full, b_full), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n", [1, 3, 8])
def test_case1_is_the_full_product(n):
    a_full = RNG.standard_normal((2 * n, 5))
    bs = [RNG.standard_normal((5, 3)) for _ in range(n)]
    out = looped.looped_allgather_einsum("mk,kn->mn", "lhs", "m", np.split(a_full, n, 0), bs)
    for r in range(n):
        np.testing.assert_allclose(out[r], oracle.einsum_bruteforce("mk,kn->mn", a_full, bs[r]), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_case3_is_the_batched_product(n):
    l_full = RNG.standard_normal((2 * n, 3, 4))
    rs = [RNG.standard_normal((2 * n, 4, 2)) for _ in range(n)]
    out = looped.looped_allgather_einsum("bmk,bkn->bmn", "lhs", "b", np.split(l_full, n, 0), rs)
    for r in range(n):
        np.testing.assert_allclose(out[r], oracle.einsum_bruteforce("bmk,bkn->bmn", l_full, rs[r]), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n", [1, 2, 3, 8])
@pytest.mark.parametrize("out_label", ["m", "n"])
def test_einsum_rs_is_a_slice_of_the_concatenated_product(n, out_label):
    # sum_q L_q @ R_q = [L_0 ... L_{n-1}] @ [R_0; ...; R_{n-1}] (block identity);
    # rank r must hold block r of it along the output dimension.
    ls = [RNG.standard_normal((2 * n, 3)) for _ in range(n)]
    rs = [RNG.standard_normal((3, 2 * n)) for _ in range(n)]
    full = oracle.einsum_bruteforce("mk,kn->mn", np.concatenate(ls, 1), np.concatenate(rs, 0))
    out = looped.looped_einsum_reduce_scatter("mk,kn->mn", ls, rs, out_label)
    blocks = np.split(full, n, axis=0 if out_label == "m" else 1)
    for r in range(n):
        np.testing.assert_allclose(out[r], blocks[r], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------- dropout hash


def test_splitmix64_published_vectors():
    with open(os.path.join(GOLDEN, "splitmix64_vectors.txt")) as f:
        rows = [tuple(map(int, l.split())) for l in f if l.strip() and not l.startswith("#")]
    seeds = {s for s, _, _ in rows}
    for seed in seeds:
        want = {i: v for s, i, v in rows if s == seed}
        got = fused.splitmix64(seed, max(want) + 1)
        for i, v in want.items():
            assert got[i] == v
        # the vectorised counter hash is the same sequence (element e = output e+1)
        vec = fused.counter_hash(seed, np.arange(max(want) + 1))
        assert [int(x) for x in vec] == got


def test_counter_hash_matches_sequence_far_out():
    seq = fused.splitmix64(0, 1000)
    assert [int(x) for x in fused.counter_hash(0, np.arange(1000))] == seq


def test_keep_threshold_closed_form():
    assert fused.keep_threshold(0.1) == 15099494  # floor(0.9f * 2^24)
    assert fused.keep_threshold(0.0) == 1 << 24
    assert fused.keep_threshold(1.0) == 0
    assert fused.keep_threshold(0.5) == 1 << 23
    with pytest.raises(ValueError):
        fused.keep_threshold(1.5)


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_fraction_within_5_sigma(p):
    n = 1 << 22
    k = fused.keep_mask(7, p, np.arange(n)).mean()
    sigma = np.sqrt(p * (1 - p) / n)
    assert abs(k - (1 - p)) < 5 * sigma


def test_keep_mask_extremes():
    idx = np.arange(10000)
    assert fused.keep_mask(3, 0.0, idx).all()
    assert not fused.keep_mask(3, 1.0, idx).any()


# ------------------------------------------------------------ fused allreduce


def _far_inputs(n=3, shape=(4, 8)):
    parts = [RNG.standard_normal(shape) for _ in range(n)]
    bias = RNG.standard_normal(shape[-1])
    res = RNG.standard_normal(shape)
    return parts, bias, res


def test_fused_without_extras_is_the_allreduce():
    parts, _, _ = _far_inputs()
    out = oracle.fused_allreduce(parts, None, None, 0.0, 0)
    assert np.array_equal(out, oracle.allreduce(parts)[0])
    zeros_b, zeros_r = np.zeros(8), np.zeros((4, 8))
    out2 = oracle.fused_allreduce(parts, zeros_b, zeros_r, 0.0, 0)
    assert np.array_equal(out2, oracle.allreduce(parts)[0])


def test_fused_p0_adds_bias_over_last_dim_and_residual():
    parts = [np.full((2, 3), 1.0), np.full((2, 3), 2.0)]
    bias = np.array([10.0, 20.0, 30.0])
    res = np.array([[100.0, 200.0, 300.0], [400.0, 500.0, 600.0]])
    out = oracle.fused_allreduce(parts, bias, res, 0.0, 0)
    assert np.array_equal(out, np.array([[113.0, 223.0, 333.0], [413.0, 523.0, 633.0]]))


def test_fused_dropped_elements_equal_residual_and_bias_is_inside_dropout():
    parts, bias, res = _far_inputs(shape=(64, 32))
    p, seed = 0.3, 11
    out = oracle.fused_allreduce(parts, bias, res, p, seed)
    keep = fused.keep_mask(seed, p, np.arange(out.size)).reshape(out.shape)
    assert (~keep).any() and keep.any()
    # dropped: exactly the residual (bias and sum were dropped with it: bias is added
    # before dropout, the residual after, [CoCoNet] Fig. 3 order)
    assert np.array_equal(out[~keep], res[~keep])
    # kept: minus the residual, the value is a multiple 1/(1-p) of (sum + bias)
    s = sum(parts) + bias
    np.testing.assert_allclose((out - res)[keep] * (1 - np.float32(p)), s[keep], rtol=1e-12, atol=1e-12)


def test_fused_mask_depends_on_element_index_only():
    # replicated outputs: the mask must not depend on anything rank-specific
    parts, bias, res = _far_inputs(n=2)
    a = oracle.fused_allreduce(parts, bias, res, 0.5, 5)
    b = oracle.fused_allreduce(parts[::-1], bias, res, 0.5, 5)
    np.testing.assert_allclose(a, b, rtol=1e-15, atol=1e-15)


# ------------------------------------------------------------- composite models


@pytest.mark.parametrize("n", [1, 2, 4])
@pytest.mark.parametrize("is_looped", [True, False])
def test_mlp_1d_megatron_reading_equals_unpartitioned(n, is_looped):
    b, f, h = 4 * n, 16, 8 * n
    x, w1, w2 = RNG.standard_normal((b, f)), RNG.standard_normal((f, h)), RNG.standard_normal((h, f))
    y = oracle.mlp_1d_forward(np.split(x, n, 0), np.split(w1, n, 1), np.split(w2, n, 0), "megatron", is_looped)
    ref = np.split(oracle.mlp_1d_reference(x, w1, w2), n, 0)
    for r in range(n):
        np.testing.assert_allclose(y[r], ref[r], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_mlp_1d_weights_gathered_reading_equals_unpartitioned(n):
    b, f, h = 4 * n, 16, 8 * n
    x, w1, w2 = RNG.standard_normal((b, f)), RNG.standard_normal((f, h)), RNG.standard_normal((h, f))
    y = oracle.mlp_1d_forward(np.split(x, n, 0), np.split(w1, n, 0), np.split(w2, n, 0), "weights_gathered")
    ref = np.split(oracle.mlp_1d_reference(x, w1, w2), n, 0)
    for r in range(n):
        np.testing.assert_allclose(y[r], ref[r], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("m_x,n_y", [(2, 4), (1, 2), (2, 1), (3, 2)])
@pytest.mark.parametrize("is_looped", [True, False])
def test_mlp_2d_equals_unpartitioned(m_x, n_y, is_looped):
    b, f, h = 2 * n_y * 2, 3 * m_x * n_y, 2 * m_x * 3
    x, w1, w2 = RNG.standard_normal((b, f)), RNG.standard_normal((f, h)), RNG.standard_normal((h, f))

    def blocks(a, rows_by, cols_by):  # rows_by / cols_by: "x" or "y"
        out = {}
        for xi in range(m_x):
            for yi in range(n_y):
                ri, nr = (xi, m_x) if rows_by == "x" else (yi, n_y)
                ci, nc = (xi, m_x) if cols_by == "x" else (yi, n_y)
                out[(xi, yi)] = np.split(np.split(a, nr, 0)[ri], nc, 1)[ci]
        return out

    y = oracle.mlp_2d_forward(blocks(x, "y", "x"), blocks(w1, "y", "x"), blocks(w2, "x", "y"), m_x, n_y, is_looped)
    ref = oracle.mlp_2d_reference(x, w1, w2, m_x, n_y)
    for key in ref:
        np.testing.assert_allclose(y[key], ref[key], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("n", [1, 2, 8])
def test_megatron_tail_is_the_full_matmul_when_extras_vanish(n):
    x, w = RNG.standard_normal((6, 4 * n)), RNG.standard_normal((4 * n, 5))
    _, out = oracle.megatron_attention_tail(np.split(x, n, 1), np.split(w, n, 0), None, None, 0.0, 0)
    np.testing.assert_allclose(out, oracle.einsum_bruteforce("mk,kn->mn", x, w), rtol=1e-12, atol=1e-12)


# --------------------------------------------- planted mistakes (CPU, oracle only)


def test_planted_reverse_permute_breaks_rs_alignment(monkeypatch):
    monkeypatch.setattr(looped, "permute_pairs", lambda n: [(s, (s + 1) % n) for s in range(n)])
    lhs = [small_ints((8, 3)) for _ in range(4)]
    rhs = [small_ints((3, 2)) for _ in range(4)]
    trace = []
    looped.looped_allgather_einsum("mk,kn->mn", "lhs", "m", [l[:2] for l in lhs], rhs, trace)
    held = {(i, r): s for i, r, s in trace}
    assert any(held[(i, r)] != (r + i) % 4 for i in range(4) for r in range(4))
    # the RS still aligns (a full circle) but the first-index rule now fails
    trace = []
    looped.looped_einsum_reduce_scatter("mk,kn->mn", lhs, rhs, "m", trace)
    sid = {(i, q): s for i, q, s in trace}
    assert [sid[(0, q)] for q in range(4)] != [(q + 1) % 4 for q in range(4)]


def test_planted_dropped_bias_term_is_caught(monkeypatch):
    real = fused.fused_allreduce

    def no_bias(partials, bias=None, residual=None, p=0.0, seed=0):
        return real(partials, None, residual, p, seed)

    parts = [np.full((2, 3), 1.0), np.full((2, 3), 2.0)]
    bias = np.array([10.0, 20.0, 30.0])
    res = np.zeros((2, 3))
    assert not np.array_equal(no_bias(parts, bias, res), np.array([[13.0, 23.0, 33.0]] * 2))
    assert np.array_equal(real(parts, bias, res), np.array([[13.0, 23.0, 33.0]] * 2))


def test_planted_transposed_operand_is_caught():
    a, b = RNG.standard_normal((3, 3)), RNG.standard_normal((3, 3))
    wrong = np.matmul(a.T, b)
    assert not np.allclose(wrong, oracle.einsum_bruteforce("mk,kn->mn", a, b))
    np.testing.assert_allclose(oracle.einsum("mk,kn->mn", a, b), oracle.einsum_bruteforce("mk,kn->mn", a, b), rtol=1e-13)


def test_planted_wrong_shard_index_in_case2_is_caught(monkeypatch):
    # DynamicSlice with the rank instead of the received shard's ID
    n = 4
    a_full, b_full = small_ints((3, 2 * n)), small_ints((2 * n, 3))
    shards = np.split(a_full, n, 1)
    good = looped.looped_allgather_einsum("mk,kn->mn", "lhs", "k", shards, [b_full] * n)
    real_slice = looped._slice
    calls = {"k": 0}

    def bad_slice(arr, dim, index, size):
        calls["k"] += 1
        return real_slice(arr, dim, 0, size)

    monkeypatch.setattr(looped, "_slice", bad_slice)
    bad = looped.looped_allgather_einsum("mk,kn->mn", "lhs", "k", shards, [b_full] * n)
    assert calls["k"] > 0
    assert any(not np.array_equal(x, y) for x, y in zip(good, bad))
    np.testing.assert_array_equal(good[0], oracle.einsum_bruteforce("mk,kn->mn", a_full, b_full))


# ------------------------------------------- schedule variants ([Decomp] §5.4)


@pytest.mark.parametrize("case", AG_CASES)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_bidirectional_allgather_einsum_equals_monolithic(case, n):
    spec, side, lab, shp, _ = case
    shards = [small_ints(shp) for _ in range(n)]
    locs = [small_ints(_other_shape(case, n)) for _ in range(n)]
    trace = []
    a = looped.looped_allgather_einsum_bidirectional(spec, side, lab, shards, locs, trace)
    b = looped.allgather_einsum(spec, side, lab, shards, locs)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # step k brings shards r+k and r-k (from the two directions); every shard is used once
    for r in range(n):
        used = [(st, s) for st, rr, s in trace if rr == r]
        assert sorted(s for _, s in used) == list(range(n))
        for st, s in used:
            assert s in ((r + st) % n, (r - st) % n)
    steps = {st for st, _, _ in trace}
    assert len(steps) == n // 2 + 1  # about half the iterations of the ring form


@pytest.mark.parametrize("out_label", ["m", "n"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_unrolled_einsum_rs_equals_monolithic(out_label, n):
    lhs = [small_ints((2 * n, 3)) for _ in range(n)]
    rhs = [small_ints((3, 2 * n)) for _ in range(n)]
    trace = []
    a = looped.looped_einsum_reduce_scatter_unrolled("mk,kn->mn", lhs, rhs, out_label, trace)
    b = looped.einsum_reduce_scatter("mk,kn->mn", lhs, rhs, out_label)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # two interleaved chains: A collects ranks r-1, r-3, ..., B ranks r-2, r-4, ...
    for r in range(n):
        ca = [q for i, q, c, s in sorted(trace) if s == r and c == "A"]
        cb = [q for i, q, c, s in sorted(trace) if s == r and c == "B"]
        assert ca == [(r - 1 - 2 * i) % n for i in range(len(ca))]
        assert cb == [(r - 2 - 2 * i) % n for i in range(len(cb))]
        assert sorted(ca + cb) == list(range(n))


@pytest.mark.parametrize("out_label", ["m", "n"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_bidirectional_einsum_rs_equals_monolithic(out_label, n):
    lhs = [small_ints((2 * n, 3)) for _ in range(n)]
    rhs = [small_ints((3, 2 * n)) for _ in range(n)]
    trace = []
    a = looped.looped_einsum_reduce_scatter_bidirectional("mk,kn->mn", lhs, rhs, out_label, trace)
    b = looped.einsum_reduce_scatter("mk,kn->mn", lhs, rhs, out_label)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    for r in range(n):
        left = [q for i, q, d, s in sorted(trace) if s == r and d == "left"]
        right = [q for i, q, d, s in sorted(trace) if s == r and d == "right"]
        assert left == [(r + len(left) - i) % n for i in range(len(left))]  # r+a, ..., r+1
        assert right == [(r - len(right) + i) % n for i in range(len(right))]  # r-b, ..., r-1
        assert abs(len(left) - len(right)) <= 1 and len(left) + len(right) == n - 1


# ----------------------------------------------------- scattered tensors ([CoCoNet])


def test_scattered_metadata_matches_the_page():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "scattered_metadata.txt")) if l.strip() and not l.startswith("#")]
    for elements, percent in rows:
        meta = oracle.scattered_metadata_bytes(int(elements))
        assert meta == 12 * -(-int(elements) // 1024)
        # as a share of the model's 16-bit storage, rounded as the page prints it
        assert round(100.0 * meta / (2 * int(elements)), 1) == float(percent)


@pytest.mark.parametrize("numels", [[0], [1], [1023, 1024, 1025], [5000, 1, 0, 2048]])
def test_scattered_buckets_cover_every_element_once(numels):
    bl = oracle.scattered_buckets(numels)
    assert all(0 < ln <= 1024 for _, _, ln in bl)
    for t, n in enumerate(numels):
        mine = [(off, ln) for tt, off, ln in bl if tt == t]
        assert len(mine) == -(-n // 1024)
        covered = sorted(i for off, ln in mine for i in range(off, off + ln))
        assert covered == list(range(n))
        assert sum(1 for _ in mine) * 12 == oracle.scattered_metadata_bytes(n)


@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_scattered_allreduce_closed_form_and_bucket_walk(n):
    shapes = [(3, 5), (1,), (2050,), (4, 300)]
    per_rank = [[np.full(s, float(r + 1)) for s in shapes] for r in range(n)]
    out = oracle.scattered_allreduce(per_rank, alpha=0.5)
    for o, s in zip(out, shapes):
        assert o.shape == s and np.all(o == 0.5 * n * (n + 1) / 2)
    rnd = [[RNG.standard_normal(s) for s in shapes] for _ in range(n)]
    a = oracle.scattered_allreduce(rnd, 0.25)
    b = oracle.scattered_allreduce_by_buckets(rnd, 0.25)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ---------------------------------------------------------------- [Decomp] §5.5 cost model

_TIMES = [0.0, 0.5, 1.0, 2.0, 3.0, 7.5]


def test_cost_model_ring_no_slower_than_the_collective_always_pays():
    # with ring_comm <= orig_comm and no prologue / epilogue, overlapping can only help:
    # comp + comm >= max(comp, ring) whichever of comp and ring is larger
    for comp in _TIMES:
        for comm in _TIMES:
            for ring in _TIMES:
                if ring <= comm:
                    assert oracle.loop_profitable(comp, comm, ring, 0.0)


def test_cost_model_half_bandwidth_ring_closed_form():
    # §5.5's concern: the ring uses one dimension of a mesh, half the bandwidth, so ring = 2 * comm.
    # Then (no epilogue) the loop pays exactly when the computation is at least the original comm.
    for comp in _TIMES:
        for comm in _TIMES:
            assert oracle.loop_profitable(comp, comm, 2.0 * comm, 0.0) == (comp >= comm)


def test_cost_model_boundary_and_special_cases():
    assert oracle.loop_profitable(4.0, 2.0, 5.0, 1.0)        # 6 >= max(4, 5) + 1: equality enables
    assert not oracle.loop_profitable(4.0, 2.0, 5.0, 1.5)    # 6 <  6.5
    assert oracle.loop_profitable(10.0, 4.0, 8.0, 1.0)       # 14 >= 11
    assert not oracle.loop_profitable(2.0, 4.0, 8.0, 0.0)    # 6 < 8
    # no communication at all: the loop pays only when its ring is free and it adds nothing
    assert oracle.loop_profitable(3.0, 0.0, 0.0, 0.0)
    assert not oracle.loop_profitable(3.0, 0.0, 0.0, 0.5)
    assert not oracle.loop_profitable(3.0, 0.0, 3.5, 0.0)
    # compute-dominated: the ring is hidden, the saving is the original comm minus the epilogue
    assert oracle.loop_profitable(100.0, 5.0, 20.0, 5.0)
    assert not oracle.loop_profitable(100.0, 5.0, 20.0, 5.01)
    with pytest.raises(ValueError):
        oracle.loop_profitable(-1.0, 0.0, 0.0, 0.0)
    with pytest.raises(ValueError):
        oracle.loop_profitable(1.0, float("nan"), 0.0, 0.0)


def test_cost_model_epilogue_is_monotone():
    # a dearer prologue / epilogue can only switch the decision from "decompose" to "keep"
    for comp in _TIMES:
        for comm in _TIMES:
            for ring in _TIMES:
                seen_false = False
                for e in _TIMES:
                    d = oracle.loop_profitable(comp, comm, ring, e)
                    assert not (seen_false and d)
                    seen_false = seen_false or not d
