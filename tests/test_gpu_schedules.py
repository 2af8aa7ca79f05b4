"""GPU parity of the Looped CollectiveEinsum schedule variants ([Decomp] §5.4).

Loop unrolling by 2 (§5.4.1) and bidirectional transfer (§5.4.2) change the
order in which shards are visited or partials collected. Each variant is
compared with the oracle's literal restatement of the same schedule: bit for
bit on small-integer inputs (every fp32 partial sum exact), and within the
16-bit bar on normal inputs.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, dev, empty_like_list, f64

pytestmark = pytest.mark.gpu

BF16, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


AG = [  # spec, looped side, slice dim, label, shard shape, other shape (n-dependent)
    ("mk,kn->mn", "lhs", 0, "m", lambda n: (136, 72), lambda n: (72, 264)),
    ("mk,kn->mn", "lhs", 1, "k", lambda n: (200, 64), lambda n: (64 * n, 136)),
    ("mk,kn->mn", "rhs", 0, "k", lambda n: (64, 136), lambda n: (200, 64 * n)),
    ("bmk,bkn->bmn", "lhs", 0, "b", lambda n: (2, 136, 64), lambda n: (2 * n, 64, 136)),
]


def ag_run(coco, case, n, sched, kind, dtype, out_dtype):
    spec, side, dim, lab, sshape, oshape = case
    shards = synth.per_rank(30, 0, n, sshape(n), dtype, kind)
    locs = synth.per_rank(30, 1, n, oshape(n), dtype, kind)
    ref_fn = oracle.looped_allgather_einsum_bidirectional if sched == coco.SCHED_BIDIRECTIONAL \
        else oracle.looped_allgather_einsum
    refs = ref_fn(spec, side, lab, [f64(x) for x in shards], [f64(x) for x in locs])
    outs = empty_like_list(n, refs[0].shape, out_dtype)
    looped = coco.sliced(dev(shards), dim)
    local = coco.local(dev(locs))
    lhs, rhs = (looped, local) if side == "lhs" else (local, looped)
    coco.coco_looped_ag_einsum_sched(spec, lhs, rhs, coco.local(outs), sched)
    coco.coco_device_status()
    return outs, refs


@pytest.mark.parametrize("case", AG)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("sched", [1, 2])
def test_allgather_schedules_exact_on_small_integers(coco, case, n, sched):
    outs, refs = ag_run(coco, case, n, sched, "smallint", BF16, F32)
    for o, r in zip(outs, refs):
        assert np.array_equal(f64(o), r)


@pytest.mark.parametrize("case", AG)
@pytest.mark.parametrize("sched", [0, 1, 2])
def test_allgather_schedules_normal_inputs(coco, case, sched):
    outs, refs = ag_run(coco, case, 4, sched, "normal", BF16, BF16)
    for o, r in zip(outs, refs):
        assert_close(o, r, BF16)


def rs_ref(coco, sched):
    return {coco.SCHED_RING: oracle.looped_einsum_reduce_scatter,
            coco.SCHED_UNROLL2: oracle.looped_einsum_reduce_scatter_unrolled,
            coco.SCHED_BIDIRECTIONAL: oracle.looped_einsum_reduce_scatter_bidirectional}[sched]


@pytest.mark.parametrize("out_label", ["m", "n"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("sched", [0, 1, 2])
@pytest.mark.parametrize("kind,dtype", [("smallint", BF16), ("normal", BF16), ("normal", F32)])
def test_reduce_scatter_schedules(coco, out_label, n, sched, kind, dtype):
    m, ks, nn = 8 * 3 * 5 * 7, 48, 8 * n * 16
    # activations scaled by 1/sqrt(K) as in the configurations, so fp32 sums stay O(1)
    lhs = synth.per_rank(31, 0, n, (m, ks), dtype, kind, std=(n * ks) ** -0.5 if kind == "normal" else 1.0)
    rhs = synth.per_rank(31, 1, n, (ks, nn), dtype, kind)
    refs = rs_ref(coco, sched)("mk,kn->mn", [f64(x) for x in lhs], [f64(x) for x in rhs], out_label)
    odt = F32 if kind == "smallint" else dtype
    outs = empty_like_list(n, refs[0].shape, odt)
    coco.coco_looped_einsum_rs_sched("mk,kn->mn", coco.sliced(dev(lhs), 1), coco.sliced(dev(rhs), 0),
                                     coco.sliced(outs, 0 if out_label == "m" else 1), sched)
    coco.coco_device_status()
    for o, r in zip(outs, refs):
        if kind == "smallint":
            assert np.array_equal(f64(o), r)
        else:
            assert_close(o, r, dtype)


def test_unknown_schedule_is_rejected(coco):
    a = dev(synth.per_rank(32, 0, 2, (64, 64), BF16))
    b = dev(synth.per_rank(32, 1, 2, (64, 64), BF16))
    o = empty_like_list(2, (128, 64), BF16)
    with pytest.raises(coco.CocoError) as e:
        coco.coco_looped_ag_einsum_sched("mk,kn->mn", coco.sliced(a, 0), coco.local(b), coco.local(o), 7)
    assert e.value.name == "COCO_ERR_VALUE"
