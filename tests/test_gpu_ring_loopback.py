"""The one-rank-per-device ring (``ring.py``) on one GPU, with every rank in this
process (LoopbackTransport: a permute is a device copy between the ranks'
buffers), its arithmetic in the library's kernels (CocoCompute).

The loops are the ones the distributed form runs; here each is compared with
the single-launch entry points (bit for bit where both sum in the same order,
or where small-integer inputs make every sum exact) and with the float64
oracle within the stated tolerances.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import coco, ring, synth
from helpers import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _dev(ts):
    return [t.to(DEV) for t in ts]


def _f64(ts):
    return [synth.as_f64(t) for t in ts]


@pytest.mark.parametrize("n", [3, 4, 8])
@pytest.mark.parametrize("k", [128, 512])
def test_case1_ring_equals_the_single_launch(n, k):
    m, nn = 192, 320  # ragged tiles (128 x 256)
    shards = synth.per_rank(301, 0, n, (m, k), torch.bfloat16, std=k ** -0.5)
    rhs = synth.per_rank(301, 1, n, (k, nn), torch.bfloat16)
    ds, dr = _dev(shards), _dev(rhs)
    out = [torch.full((n * m, nn), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    trace = []
    ring.looped_allgather_einsum("mk,kn->mn", "lhs", "m", ds, dr, out, ring.LoopbackTransport(n),
                                 ring.CocoCompute(), trace)
    ref = [torch.empty_like(o) for o in out]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(ds, 0), coco.local(dr), coco.local(ref))
    coco.coco_device_status()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
    want = oracle.looped_allgather_einsum("mk,kn->mn", "lhs", "m", _f64(shards), _f64(rhs))
    for o, w in zip(out, want):
        assert_close(o, w, torch.bfloat16, "ring case 1")
    assert sorted(trace) == sorted((i, r, (r + i) % n) for i in range(n) for r in range(n))


@pytest.mark.parametrize("n", [4, 8])
def test_case2_ring_adds_exactly(n):
    m, ks, nn = 256, 64, 256
    shards = synth.per_rank(302, 0, n, (m, ks), torch.bfloat16, "smallint")
    rhs = synth.per_rank(302, 1, n, (n * ks, nn), torch.bfloat16, "smallint")
    ds, dr = _dev(shards), _dev(rhs)
    out = [torch.empty((m, nn), dtype=torch.float32, device=DEV) for _ in range(n)]
    ring.looped_allgather_einsum("mk,kn->mn", "lhs", "k", ds, dr, out, ring.LoopbackTransport(n), ring.CocoCompute())
    ref = [torch.empty_like(o) for o in out]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(ds, 1), coco.local(dr), coco.local(ref))
    coco.coco_device_status()
    want = oracle.looped_allgather_einsum("mk,kn->mn", "lhs", "k", _f64(shards), _f64(rhs))
    for a, b, w in zip(out, ref, want):
        assert torch.equal(a, b)
        assert np.array_equal(synth.as_f64(a), w)  # every partial sum is an exact small integer


@pytest.mark.parametrize("n", [4, 8])
def test_case3_ring_equals_the_single_launch(n):
    b, m, k, nn = 2, 256, 128, 256
    shards = synth.per_rank(303, 0, n, (b, m, k), torch.bfloat16)
    rhs = synth.per_rank(303, 1, n, (n * b, k, nn), torch.bfloat16)
    ds, dr = _dev(shards), _dev(rhs)
    out = [torch.empty((n * b, m, nn), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    ring.looped_allgather_einsum("bmk,bkn->bmn", "lhs", "b", ds, dr, out, ring.LoopbackTransport(n),
                                 ring.CocoCompute())
    ref = [torch.empty_like(o) for o in out]
    coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.sliced(ds, 0), coco.local(dr), coco.local(ref))
    coco.coco_device_status()
    want = oracle.looped_allgather_einsum("bmk,bkn->bmn", "lhs", "b", _f64(shards), _f64(rhs))
    for a, r, w in zip(out, ref, want):
        assert torch.equal(a, r)
        assert_close(a, w, torch.bfloat16, "ring case 3")


def test_gate_keeps_the_original_allgather_then_einsum():
    n, m, k, nn = 4, 128, 128, 256
    shards = synth.per_rank(304, 0, n, (m, k), torch.bfloat16)
    rhs = synth.per_rank(304, 1, n, (k, nn), torch.bfloat16)
    ds, dr = _dev(shards), _dev(rhs)
    T, C = ring.LoopbackTransport(n), ring.CocoCompute()
    looped = [torch.empty((n * m, nn), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    kept = [torch.empty_like(o) for o in looped]
    ring.looped_allgather_einsum("mk,kn->mn", "lhs", "m", ds, dr, looped, T, C, gate=(2.0, 1.0, 1.0, 0.0))
    ring.looped_allgather_einsum("mk,kn->mn", "lhs", "m", ds, dr, kept, T, C, gate=(1.0, 1.0, 5.0, 0.0))
    torch.cuda.synchronize()
    for a, b in zip(looped, kept):
        assert torch.equal(a, b)  # one M=128 tile row per shard: the same tiles either way


@pytest.mark.parametrize("n", [3, 4, 8])
def test_reduce_scatter_ring_adds_exactly(n):
    ms, k, nn = 128, 192, 256
    lhs = synth.per_rank(305, 0, n, (n * ms, k), torch.bfloat16, "smallint")
    rhs = synth.per_rank(305, 1, n, (k, nn), torch.bfloat16, "smallint")
    dl, dr = _dev(lhs), _dev(rhs)
    out = [torch.empty((ms, nn), dtype=torch.float32, device=DEV) for _ in range(n)]
    trace = []
    ring.looped_einsum_reduce_scatter("mk,kn->mn", dl, dr, out, ring.LoopbackTransport(n), ring.CocoCompute(), trace)
    ref = [torch.empty_like(o) for o in out]
    coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(dl, 1), coco.sliced(dr, 0), coco.sliced(ref, 0))
    coco.coco_device_status()
    otrace = []
    want = oracle.looped_einsum_reduce_scatter("mk,kn->mn", _f64(lhs), _f64(rhs), "m", otrace)
    for a, b, w in zip(out, ref, want):
        assert torch.equal(a, b)
        assert np.array_equal(synth.as_f64(a), w)
    assert sorted(trace) == sorted(otrace)


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_split_fused_allreduce_is_bit_identical(dtype):
    n, rows, h = 8, 64, 512
    parts = synth.per_rank(306, 0, n, (rows, h), dtype)
    bias = synth.tensor(synth.seed_of(306, 1), (h,), dtype, std=0.02)
    res = synth.tensor(synth.seed_of(306, 2), (rows, h), dtype)
    dp, db, dres = _dev(parts), bias.to(DEV), res.to(DEV)
    out = [torch.empty((rows, h), dtype=dtype, device=DEV) for _ in range(n)]
    ring.fused_allreduce(dp, db, [dres] * n, 0.1, 99, out, ring.LoopbackTransport(n), ring.CocoCompute())
    ref = [torch.empty_like(o) for o in out]
    coco.coco_fused_allreduce(coco.local(dp), db, coco.replicated([dres] * n), 0.1, 99, coco.replicated(ref))
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
    want = oracle.fused_allreduce(_f64(parts), synth.as_f64(bias), synth.as_f64(res), 0.1, 99)
    assert_close(out[0], want, dtype, "split FusedAllReduce")


def test_reduce_scatter_gate_keeps_the_original_einsum_then_reduce_scatter():
    n, ms, k, nn = 4, 128, 192, 256
    lhs = [t.to(DEV) for t in synth.per_rank(307, 0, n, (n * ms, k), torch.bfloat16, "smallint")]
    rhs = [t.to(DEV) for t in synth.per_rank(307, 1, n, (k, nn), torch.bfloat16, "smallint")]
    T, C = ring.LoopbackTransport(n), ring.CocoCompute()
    looped = [torch.empty((ms, nn), dtype=torch.float32, device=DEV) for _ in range(n)]
    kept = [torch.empty_like(o) for o in looped]
    ring.looped_einsum_reduce_scatter("mk,kn->mn", lhs, rhs, looped, T, C, gate=(2.0, 1.0, 1.0, 0.0))
    ring.looped_einsum_reduce_scatter("mk,kn->mn", lhs, rhs, kept, T, C, gate=(1.0, 1.0, 5.0, 0.0))
    torch.cuda.synchronize()
    for a, b in zip(looped, kept):
        assert torch.equal(a, b)  # small integers: every sum exact in either order


def test_case3_ring_with_the_looped_operand_on_the_right():
    n, b, m, k, nn = 4, 2, 256, 128, 256
    lhs = [t.to(DEV) for t in synth.per_rank(308, 0, n, (n * b, m, k), torch.bfloat16)]
    shards = [t.to(DEV) for t in synth.per_rank(308, 1, n, (b, k, nn), torch.bfloat16)]
    out = [torch.empty((n * b, m, nn), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    ring.looped_allgather_einsum("bmk,bkn->bmn", "rhs", "b", shards, lhs, out, ring.LoopbackTransport(n),
                                 ring.CocoCompute())
    ref = [torch.empty_like(o) for o in out]
    coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.local(lhs), coco.sliced(shards, 0), coco.local(ref))
    coco.coco_device_status()
    want = oracle.looped_allgather_einsum("bmk,bkn->bmn", "rhs", "b", _f64(shards), _f64(lhs))
    for a, r, w in zip(out, ref, want):
        assert torch.equal(a, r)
        assert_close(a, w, torch.bfloat16, "ring case 3, looped RHS")


@pytest.mark.parametrize("n", [2, 3, 4, 5, 8])
def test_bidirectional_allgather_einsum_ring(n):
    """[Decomp] section 5.4.2 with real transfers (loopback): the own shard, then r+k and r-k per step;
    the same shard order as coco_looped_ag_einsum_sched, so case 1 (DynamicUpdateSlice) is bit-equal
    and case 2 (Addition, small integers) exact."""
    m, k, nn = 128, 128, 256
    shards = [t.to(DEV) for t in synth.per_rank(309, 0, n, (m, k), torch.bfloat16, "smallint")]
    rhs = [t.to(DEV) for t in synth.per_rank(309, 1, n, (k, nn), torch.bfloat16, "smallint")]
    out = [torch.empty((n * m, nn), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    trace = []
    ring.looped_allgather_einsum("mk,kn->mn", "lhs", "m", shards, rhs, out, ring.LoopbackTransport(n),
                                 ring.CocoCompute(), trace, schedule=coco.SCHED_BIDIRECTIONAL)
    ref = [torch.empty_like(o) for o in out]
    coco.coco_looped_ag_einsum_sched("mk,kn->mn", coco.sliced(shards, 0), coco.local(rhs), coco.local(ref),
                                     coco.SCHED_BIDIRECTIONAL)
    coco.coco_device_status()
    otrace = []
    want = oracle.looped_allgather_einsum_bidirectional("mk,kn->mn", "lhs", "m", _f64(shards), _f64(rhs), otrace)
    for a, b, w in zip(out, ref, want):
        assert torch.equal(a, b)
        assert_close(a, w, torch.bfloat16, "bidirectional case 1")
    assert sorted(trace) == sorted(otrace)
    # case 2: Addition in the bidirectional order
    ks = 64
    shards2 = [t.to(DEV) for t in synth.per_rank(309, 2, n, (m, ks), torch.bfloat16, "smallint")]
    rhs2 = [t.to(DEV) for t in synth.per_rank(309, 3, n, (n * ks, nn), torch.bfloat16, "smallint")]
    out2 = [torch.empty((m, nn), dtype=torch.float32, device=DEV) for _ in range(n)]
    ring.looped_allgather_einsum("mk,kn->mn", "lhs", "k", shards2, rhs2, out2, ring.LoopbackTransport(n),
                                 ring.CocoCompute(), schedule=coco.SCHED_BIDIRECTIONAL)
    want2 = oracle.looped_allgather_einsum_bidirectional("mk,kn->mn", "lhs", "k", _f64(shards2), _f64(rhs2))
    torch.cuda.synchronize()
    for a, w in zip(out2, want2):
        assert np.array_equal(synth.as_f64(a), w)


@pytest.mark.parametrize("sched", [1, 2])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_reduce_scatter_ring_schedules(sched, n):
    """Unroll-by-2 (section 5.4.1) and bidirectional (section 5.4.2) Einsum-ReduceScatter with real
    transfers (loopback): small-integer inputs, so every sum is exact and equal to the single-launch
    schedule's and the oracle's."""
    ms, k, nn = 128, 128, 256
    lhs = [t.to(DEV) for t in synth.per_rank(310, 0, n, (n * ms, k), torch.bfloat16, "smallint")]
    rhs = [t.to(DEV) for t in synth.per_rank(310, 1, n, (k, nn), torch.bfloat16, "smallint")]
    out = [torch.empty((ms, nn), dtype=torch.float32, device=DEV) for _ in range(n)]
    trace = []
    ring.looped_einsum_reduce_scatter("mk,kn->mn", lhs, rhs, out, ring.LoopbackTransport(n), ring.CocoCompute(),
                                      trace, schedule=sched)
    ref = [torch.empty_like(o) for o in out]
    coco.coco_looped_einsum_rs_sched("mk,kn->mn", coco.sliced(lhs, 1), coco.sliced(rhs, 0), coco.sliced(ref, 0),
                                     sched)
    coco.coco_device_status()
    fn = oracle.looped_einsum_reduce_scatter_unrolled if sched == 1 else oracle.looped_einsum_reduce_scatter_bidirectional
    otrace = []
    want = fn("mk,kn->mn", _f64(lhs), _f64(rhs), "m", otrace)
    for a, b, w in zip(out, ref, want):
        assert torch.equal(a, b)
        assert np.array_equal(synth.as_f64(a), w)
    assert sorted(trace) == sorted(otrace)


@pytest.mark.parametrize("sched", [coco.SCHED_RING, coco.SCHED_UNROLL2])
def test_compute_on_its_own_stream_is_ordered_with_the_transfers(sched):
    # The transfers (device copies here, torch.distributed between devices) are ordered on the current
    # stream; kernels on a side stream are joined to it around every call, so the loop gives the same
    # bits as on the current stream.
    n, m, k, nn = 4, 256, 256, 256
    hl = synth.per_rank(311, 0, n, (n * m, k), torch.bfloat16, "smallint")
    hr = synth.per_rank(311, 1, n, (k, nn), torch.bfloat16, "smallint")
    lhs, rhs = _dev(hl), _dev(hr)
    side = torch.cuda.Stream(device=DEV)
    outs = []
    for compute in (ring.CocoCompute(), ring.CocoCompute(stream=side)):
        out = [torch.full((m, nn), float("nan"), dtype=torch.float32, device=DEV) for _ in range(n)]
        ring.looped_einsum_reduce_scatter("mk,kn->mn", lhs, rhs, out, ring.LoopbackTransport(n), compute,
                                          schedule=sched)
        outs.append(out)
    torch.cuda.synchronize()
    coco.coco_device_status()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    want = oracle.looped_einsum_reduce_scatter("mk,kn->mn", _f64(hl), _f64(hr), "m")
    for o, w in zip(outs[1], want):
        assert np.array_equal(synth.as_f64(o), w)
