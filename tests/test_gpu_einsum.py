"""GPU parity of the looped einsums against the oracle, through the C-ABI.

Looped AllGather-Einsum cases 1, 2 and 3 (and their mirrored forms with the
looped operand on the right), Looped Einsum-ReduceScatter on either output
dimension, and the local MatMul ([Decomp] §5.1; [CoCoNet] Fig. 3). bf16 / f16
run on the tcgen05 path, fp32 on the FMA path. Sizes span several 128 x 256
tiles with ragged M, N and K tails.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, dev, empty_like_list, f64

pytestmark = pytest.mark.gpu

BF16, F16, F32 = torch.bfloat16, torch.float16, torch.float32
IN_DTYPES = [BF16, F16, F32]


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


def gen(cfg, tid, n, shape, dtype, kind="normal", std=1.0):
    return synth.per_rank(cfg, tid, n, shape, dtype, kind, std)


def check(coco, outs, refs, out_dtype, what):
    coco.coco_device_status()
    torch.cuda.synchronize()
    for r, (o, ref) in enumerate(zip(outs, refs)):
        assert_close(o, ref, out_dtype, f"{what} rank {r}")


@pytest.mark.parametrize("dtype", IN_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_case1_lhs_sliced_on_rows(coco, dtype, n):
    ms, k, nn = 136, 200, 264
    shards = gen(11, 0, n, (ms, k), dtype, std=k ** -0.5)
    rhs = gen(11, 1, n, (k, nn), dtype)
    outs = empty_like_list(n, (n * ms, nn), dtype)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 0), coco.local(dev(rhs)), coco.local(outs))
    refs = oracle.allgather_einsum("mk,kn->mn", "lhs", "m", [f64(s) for s in shards], [f64(x) for x in rhs])
    check(coco, outs, refs, dtype, "case 1")


@pytest.mark.parametrize("dtype,out_dtype", [(BF16, F32), (BF16, BF16), (F16, F32), (F32, F32), (F16, F16)])
@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_case2_lhs_sliced_on_k(coco, dtype, out_dtype, n):
    m, ks, nn = 300, 40, 264
    shards = gen(12, 0, n, (m, ks), dtype, std=(n * ks) ** -0.5)
    rhs = gen(12, 1, n, (n * ks, nn), dtype)
    outs = empty_like_list(n, (m, nn), out_dtype)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 1), coco.local(dev(rhs)), coco.local(outs))
    refs = oracle.allgather_einsum("mk,kn->mn", "lhs", "k", [f64(s) for s in shards], [f64(x) for x in rhs])
    check(coco, outs, refs, out_dtype, "case 2")


@pytest.mark.parametrize("dtype", IN_DTYPES)
@pytest.mark.parametrize("n", [2, 3, 8])
def test_case2_rhs_sliced_on_k(coco, dtype, n):
    m, ks, nn = 264, 72, 136
    lhs = gen(13, 0, n, (m, n * ks), dtype, std=(n * ks) ** -0.5)
    shards = gen(13, 1, n, (ks, nn), dtype)
    outs = empty_like_list(n, (m, nn), dtype)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.local(dev(lhs)), coco.sliced(dev(shards), 0), coco.local(outs))
    refs = oracle.allgather_einsum("mk,kn->mn", "rhs", "k", [f64(s) for s in shards], [f64(x) for x in lhs])
    check(coco, outs, refs, dtype, "case 2 mirrored")


@pytest.mark.parametrize("dtype", IN_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 4])
def test_case1_rhs_sliced_on_cols(coco, dtype, n):
    m, k, ns = 200, 136, 264
    lhs = gen(14, 0, n, (m, k), dtype, std=k ** -0.5)
    shards = gen(14, 1, n, (k, ns), dtype)
    outs = empty_like_list(n, (m, n * ns), dtype)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.local(dev(lhs)), coco.sliced(dev(shards), 1), coco.local(outs))
    refs = oracle.allgather_einsum("mk,kn->mn", "rhs", "n", [f64(s) for s in shards], [f64(x) for x in lhs])
    check(coco, outs, refs, dtype, "case 1 mirrored")


@pytest.mark.parametrize("dtype", IN_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 4])
def test_case3_lhs_sliced_on_batch(coco, dtype, n):
    bs, m, k, nn = 2, 136, 72, 264
    shards = gen(15, 0, n, (bs, m, k), dtype, std=k ** -0.5)
    rhs = gen(15, 1, n, (n * bs, k, nn), dtype)
    outs = empty_like_list(n, (n * bs, m, nn), dtype)
    coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.sliced(dev(shards), 0), coco.local(dev(rhs)),
                               coco.local(outs))
    refs = oracle.allgather_einsum("bmk,bkn->bmn", "lhs", "b", [f64(s) for s in shards], [f64(x) for x in rhs])
    check(coco, outs, refs, dtype, "case 3")


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("label,dim", [("b", 0), ("m", 1), ("k", 2)])
def test_batched_rhs_and_lhs_variants(coco, dtype, label, dim):
    n, b, m, k, nn = 2, 4, 136, 80, 136
    lshape = [b, m, k]
    lshape[dim] //= n
    shards = gen(16, 0, n, tuple(lshape), dtype, std=k ** -0.5)
    rhs = gen(16, 1, n, (b, k, nn), dtype)
    outs = empty_like_list(n, (b, m, nn), dtype)
    coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.sliced(dev(shards), dim), coco.local(dev(rhs)),
                               coco.local(outs))
    refs = oracle.allgather_einsum("bmk,bkn->bmn", "lhs", label, [f64(s) for s in shards], [f64(x) for x in rhs])
    check(coco, outs, refs, dtype, f"batched lhs sliced on {label}")
    # the mirrored batched case 3: rhs sliced on batch
    lhs = gen(16, 2, n, (b, m, k), dtype, std=k ** -0.5)
    rsh = gen(16, 3, n, (b // n, k, nn), dtype)
    outs = empty_like_list(n, (b, m, nn), dtype)
    coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.local(dev(lhs)), coco.sliced(dev(rsh), 0), coco.local(outs))
    refs = oracle.allgather_einsum("bmk,bkn->bmn", "rhs", "b", [f64(s) for s in rsh], [f64(x) for x in lhs])
    check(coco, outs, refs, dtype, "batched rhs sliced on b")


@pytest.mark.parametrize("dtype", IN_DTYPES)
@pytest.mark.parametrize("out_label", ["m", "n"])
@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_looped_einsum_reduce_scatter(coco, dtype, out_label, n):
    m, ks, nn = 408, 48, 384  # 408 rows split into 1/2/3/8 shards; 384 / n is a multiple of 8
    lhs = gen(17, 0, n, (m, ks), dtype, std=(n * ks) ** -0.5)
    rhs = gen(17, 1, n, (ks, nn), dtype)
    oshape = (m // n, nn) if out_label == "m" else (m, nn // n)
    outs = empty_like_list(n, oshape, dtype)
    coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(dev(lhs), 1), coco.sliced(dev(rhs), 0),
                               coco.sliced(outs, 0 if out_label == "m" else 1))
    refs = oracle.einsum_reduce_scatter("mk,kn->mn", [f64(x) for x in lhs], [f64(x) for x in rhs], out_label)
    check(coco, outs, refs, dtype, f"einsum-rs on {out_label}")


@pytest.mark.parametrize("dtype,out_dtype", [(F16, F16), (BF16, BF16), (F32, F32), (BF16, F32)])
def test_local_matmul_of_k_sliced_operands(coco, dtype, out_dtype):
    n, m, ks, nn = 4, 264, 64, 520
    lhs = gen(18, 0, n, (m, ks), dtype)
    rhs = gen(18, 1, n, (ks, nn), dtype, std=0.02)
    outs = empty_like_list(n, (m, nn), out_dtype)
    coco.coco_einsum("mk,kn->mn", coco.sliced(dev(lhs), 1), coco.sliced(dev(rhs), 0), coco.local(outs))
    refs = [oracle.einsum("mk,kn->mn", f64(a), f64(b)) for a, b in zip(lhs, rhs)]
    check(coco, outs, refs, out_dtype, "local matmul")


def test_replicated_local_operand_gives_replicated_output(coco):
    n, ms, k, nn = 4, 64, 64, 256
    shards = gen(19, 0, n, (ms, k), BF16, std=k ** -0.5)
    w = gen(19, 1, 1, (k, nn), BF16)[0].cuda()
    outs = empty_like_list(n, (n * ms, nn), BF16)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 0), coco.replicated([w] * n),
                               coco.replicated(outs))
    ref = oracle.allgather_einsum("mk,kn->mn", "lhs", "m", [f64(s) for s in shards], [f64(w)])[0]
    check(coco, outs, [ref] * n, BF16, "replicated")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_groups_run_independently(coco):
    g, n, ms, k, nn = 3, 2, 128, 64, 256
    shards = gen(20, 0, g * n, (ms, k), BF16, std=k ** -0.5)
    rhs = gen(20, 1, g * n, (k, nn), BF16)
    outs = empty_like_list(g * n, (n * ms, nn), BF16)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 0, ngroups=g), coco.local(dev(rhs), ngroups=g),
                               coco.local(outs, ngroups=g))
    coco.coco_device_status()
    for gi in range(g):
        sl = slice(gi * n, (gi + 1) * n)
        refs = oracle.allgather_einsum("mk,kn->mn", "lhs", "m", [f64(s) for s in shards[sl]],
                                       [f64(x) for x in rhs[sl]])
        for r in range(n):
            assert_close(outs[gi * n + r], refs[r], BF16, f"group {gi} rank {r}")


@pytest.mark.parametrize("dtype", [BF16, F16, F32])
def test_small_integers_are_exact(coco, dtype):
    # |v| <= 4 and K*16 < 2^24: every partial sum is exact in fp32, so the GPU's
    # ring-order accumulation must equal the oracle bit for bit (looped == monolithic).
    n, m, ks, nn = 4, 136, 64, 264
    shards = gen(21, 0, n, (m, ks), dtype, "smallint")
    rhs = gen(21, 1, n, (n * ks, nn), dtype, "smallint")
    outs = empty_like_list(n, (m, nn), F32)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 1), coco.local(dev(rhs)), coco.local(outs))
    coco.coco_device_status()
    refs = oracle.looped_allgather_einsum("mk,kn->mn", "lhs", "k", [f64(s) for s in shards], [f64(x) for x in rhs])
    for o, ref in zip(outs, refs):
        assert np.array_equal(f64(o), ref)
    lhs = gen(21, 2, n, (n * 16, ks), dtype, "smallint")
    rhs2 = gen(21, 3, n, (ks, nn), dtype, "smallint")
    outs = empty_like_list(n, (16, nn), F32)
    coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(dev(lhs), 1), coco.sliced(dev(rhs2), 0), coco.sliced(outs, 0))
    coco.coco_device_status()
    refs = oracle.looped_einsum_reduce_scatter("mk,kn->mn", [f64(x) for x in lhs], [f64(x) for x in rhs2], "m")
    for o, ref in zip(outs, refs):
        assert np.array_equal(f64(o), ref)


def test_zero_contraction_gives_zeros(coco):
    n = 2
    lhs = [torch.empty((0, 0), dtype=BF16, device="cuda") for _ in range(n)]
    a = coco.Dist(coco.SLICED, lhs, (64, 0), slice_dim=1)
    b = coco.Dist(coco.LOCAL, [torch.empty((0, 64), dtype=BF16, device="cuda") for _ in range(n)], (0, 64))
    outs = [torch.full((64, 64), 3.0, dtype=BF16, device="cuda") for _ in range(n)]
    coco.coco_looped_ag_einsum("mk,kn->mn", a, b, coco.local(outs))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.count_nonzero(o) == 0


@pytest.mark.parametrize("n,g", [(64, 1), (32, 2), (40, 1)])
def test_looped_einsums_at_the_pointer_limit(coco, n, g):
    """Up to 64 ranks (or 32 x 2 groups): the planner spreads the N x N (rank, step) jobs of case 1 and
    their operand maps over several launches. The einsum-ReduceScatter sums N rank slices per output
    region, two operand views each, which one launch holds up to N = 40; beyond that the call returns
    COCO_ERR_UNSUPPORTED and launches nothing."""
    ms, k, nn = 16, 64, 64
    shards = gen(40, 0, n * g, (ms, k), BF16, std=k ** -0.5)
    rhs = gen(40, 1, n * g, (k, nn), BF16)
    outs = empty_like_list(n * g, (n * ms, nn), BF16)
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 0, ngroups=g), coco.local(dev(rhs), ngroups=g),
                               coco.local(outs, ngroups=g))
    for gi in range(g):
        sl = slice(gi * n, (gi + 1) * n)
        refs = oracle.allgather_einsum("mk,kn->mn", "lhs", "m", [f64(s) for s in shards[sl]],
                                       [f64(x) for x in rhs[sl]])
        check(coco, outs[sl], refs, BF16, f"case 1 group {gi}")
    ks = 16
    lhs = gen(41, 0, n * g, (ms, ks), BF16, std=(n * ks) ** -0.5)
    rw = gen(41, 1, n * g, (ks, n * 8), BF16)
    ys = empty_like_list(n * g, (ms, 8), BF16)
    if n > 40:
        with pytest.raises(coco.CocoError) as exc:
            coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(dev(lhs), 1, ngroups=g),
                                       coco.sliced(dev(rw), 0, ngroups=g), coco.sliced(ys, 1, ngroups=g))
        assert exc.value.name == "COCO_ERR_UNSUPPORTED"
        torch.cuda.synchronize()
        assert all(torch.isnan(y).all() for y in ys)  # nothing ran
        return
    coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(dev(lhs), 1, ngroups=g), coco.sliced(dev(rw), 0, ngroups=g),
                               coco.sliced(ys, 1, ngroups=g))
    for gi in range(g):
        sl = slice(gi * n, (gi + 1) * n)
        refs = oracle.einsum_reduce_scatter("mk,kn->mn", [f64(x) for x in lhs[sl]], [f64(x) for x in rw[sl]], "n")
        check(coco, ys[sl], refs, BF16, f"einsum-RS group {gi}")

