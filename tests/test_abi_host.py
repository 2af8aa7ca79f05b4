"""Host-side tests of the C-ABI: the library loads, exports every symbol the
header declares, and rejects invalid arguments before any CUDA call.

These run without a GPU: all device pointers are fake addresses that the
library validates but never dereferences, and every case returns before the
first CUDA call (an error status, or COCO_OK for an empty tensor).
"""

import ctypes
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def coco():
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


def header_functions():
    text = open(os.path.join(ROOT, "include", "coco.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(coco_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for want in ["coco_fused_allreduce", "coco_allreduce_rs_ag", "coco_allgather", "coco_reduce_scatter",
                 "coco_allreduce", "coco_looped_ag_einsum", "coco_looped_einsum_rs", "coco_einsum",
                 "coco_status_string"]:
        assert want in names


def test_library_exports_every_declared_symbol(coco):
    lib = ctypes.CDLL(coco.library_path())
    for name in header_functions():
        assert hasattr(lib, name), name
    assert sorted(coco.EXPORTED) == header_functions()


def test_status_strings(coco):
    for code, name in coco.STATUS.items():
        assert coco._lib.coco_status_string(code).decode().startswith(name)
    assert coco.version() >= 100


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def mk(coco, dtype, layout, shape, nranks, ngroups=1, slice_dim=-1, base=FAKE, stride=1 << 32, ptrs=None):
    t = coco.CocoTensor()
    t.dtype, t.layout, t.ndim, t.slice_dim = dtype, layout, len(shape), slice_dim
    for i, s in enumerate(shape):
        t.shape[i] = s
    t.nranks, t.ngroups = nranks, ngroups
    for i in range(min(nranks * ngroups, coco.MAX_PTRS)):
        t.ptr[i] = ptrs[i] if ptrs is not None else base + i * stride
    return t


def far(coco, partials, out, residual=None, bias=None, p=0.0):
    return coco.raw_call("coco_fused_allreduce", ctypes.byref(partials), bias,
                         None if residual is None else ctypes.byref(residual), p, 0, ctypes.byref(out), None)


def test_far_validation(coco):
    F16, L, R, S = coco.F16, coco.LOCAL, coco.REPLICATED, coco.SLICED
    good_in = mk(coco, F16, L, (4, 16), 2)
    good_out = mk(coco, F16, R, (4, 16), 2, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_fused_allreduce", None, None, None, 0.0, 0, ctypes.byref(good_out), None) == 1
    # layouts
    assert far(coco, mk(coco, F16, R, (4, 16), 2), good_out) == 4
    assert far(coco, good_in, mk(coco, F16, L, (4, 16), 2, base=FAKE + (1 << 40))) == 4
    # dtypes
    assert far(coco, good_in, mk(coco, coco.BF16, R, (4, 16), 2, base=FAKE + (1 << 40))) == 3
    bad = mk(coco, F16, L, (4, 16), 2)
    bad.dtype = 7
    assert far(coco, bad, good_out) == 3
    # shapes / ranks
    assert far(coco, good_in, mk(coco, F16, R, (4, 24), 2, base=FAKE + (1 << 40))) == 2
    assert far(coco, good_in, mk(coco, F16, R, (4, 16), 4, base=FAKE + (1 << 40))) == 2
    bad = mk(coco, F16, L, (4, 16), 2)
    bad.ndim = 4
    assert far(coco, bad, good_out) == 2
    bad = mk(coco, F16, L, (4, 16), 33, ngroups=2)
    assert far(coco, bad, good_out) == 2
    # alignment: pointer and inner dimension
    assert far(coco, mk(coco, F16, L, (4, 16), 2, base=FAKE + 8), good_out) == 5
    assert far(coco, mk(coco, F16, L, (4, 12), 2), mk(coco, F16, R, (4, 12), 2, base=FAKE + (1 << 40))) == 5
    assert far(coco, good_in, good_out, bias=ctypes.c_void_p(FAKE + (1 << 41) + 4)) == 5
    # null pointers
    assert far(coco, mk(coco, F16, L, (4, 16), 2, ptrs=[FAKE, 0]), good_out) == 1
    # dropout probability
    assert far(coco, good_in, good_out, p=1.5) == 10
    assert far(coco, good_in, good_out, p=-0.1) == 10
    assert far(coco, good_in, good_out, p=float("nan")) == 10
    # residual
    assert far(coco, good_in, good_out, residual=mk(coco, F16, L, (4, 16), 2, base=FAKE + (1 << 42))) == 4
    assert far(coco, good_in, good_out, residual=mk(coco, F16, R, (8, 16), 2, base=FAKE + (1 << 42))) == 2
    # more than 2^40 elements per rank is refused before any size is computed from it (no overflow)
    huge = (1 << 40, 1 << 40, 16)
    assert far(coco, mk(coco, F16, L, huge, 2), mk(coco, F16, R, huge, 2, base=FAKE + (1 << 40))) == 2
    assert far(coco, mk(coco, F16, L, (1 << 20, 1 << 20, 16), 2),
               mk(coco, F16, R, (1 << 20, 1 << 20, 16), 2, base=FAKE + (1 << 40))) == 2


def test_far_at_index_base_validation(coco):
    """coco_fused_allreduce_at: index_base must be a multiple of the 16-byte vector width in elements;
    the other checks are coco_fused_allreduce's."""
    F16, F32, L, R = coco.F16, coco.F32, coco.LOCAL, coco.REPLICATED

    def far_at(dtype, base, p=0.0):
        ins = mk(coco, dtype, L, (4, 16), 2)
        outs = mk(coco, dtype, R, (4, 16), 2, base=FAKE + (1 << 40))
        return coco.raw_call("coco_fused_allreduce_at", ctypes.byref(ins), None, None, p, 0, base,
                             ctypes.byref(outs), None)

    assert far_at(F16, 4) == 5   # 16-bit: multiples of 8 elements
    assert far_at(F16, 12) == 5
    assert far_at(F32, 2) == 5   # fp32: multiples of 4
    assert far_at(F16, 16, p=2.0) == 10  # the shared checks still apply
    empty_in = mk(coco, F16, L, (0, 16), 2)
    empty_out = mk(coco, F16, R, (0, 16), 2, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_fused_allreduce_at", ctypes.byref(empty_in), None, None, 0.1, 0, 8 * 1000,
                         ctypes.byref(empty_out), None) == 0


def test_wait_selftest_limit_validation(coco):
    for bad in (0, 999, 1_000_000_001, 2 ** 63):
        assert coco.raw_call("coco_wait_selftest", bad, None) == 10


def test_far_aliasing(coco):
    F16, L, R = coco.F16, coco.LOCAL, coco.REPLICATED
    nbytes = 4 * 16 * 2
    ins = mk(coco, F16, L, (4, 16), 2, stride=1 << 20)
    # output shifted into the middle of an input: partial overlap
    out = mk(coco, F16, R, (4, 16), 2, ptrs=[FAKE + 16, FAKE + (1 << 30)])
    assert far(coco, ins, out) == 6
    # two distinct outputs overlapping each other
    out = mk(coco, F16, R, (4, 16), 2, ptrs=[FAKE + (1 << 30), FAKE + (1 << 30) + 32])
    assert far(coco, ins, out) == 6
    # bias inside an output
    out = mk(coco, F16, R, (4, 16), 2, ptrs=[FAKE + (1 << 30)] * 2)
    assert far(coco, ins, out, bias=ctypes.c_void_p(FAKE + (1 << 30) + 32)) == 6
    assert nbytes > 32


def test_empty_tensors_return_ok_without_cuda(coco):
    F32, L, R, S = coco.F32, coco.LOCAL, coco.REPLICATED, coco.SLICED
    e_in = mk(coco, F32, L, (0, 16), 2)
    e_out = mk(coco, F32, R, (0, 16), 2, base=FAKE + (1 << 40))
    assert far(coco, e_in, e_out) == 0
    assert coco.raw_call("coco_allreduce", ctypes.byref(e_in), ctypes.byref(e_out), None) == 0
    e_sl = mk(coco, F32, S, (0, 16), 2, slice_dim=0, base=FAKE + (1 << 41))
    assert coco.raw_call("coco_reduce_scatter", ctypes.byref(e_in), ctypes.byref(e_sl), None) == 0
    assert coco.raw_call("coco_allgather", ctypes.byref(e_sl), ctypes.byref(e_out), None) == 0
    assert coco.raw_call("coco_dropout_keep_mask", 0, ctypes.c_float(0.1), 0, 0, None, None) == 0
    assert coco.raw_call("coco_dropout_keep_mask", 0, ctypes.c_float(0.1), 0, 5, None, None) == 1
    # einsum with an empty output
    lhs = mk(coco, F32, S, (0, 16), 2, slice_dim=0)
    rhs = mk(coco, F32, L, (16, 8), 2, base=FAKE + (1 << 41))
    out = mk(coco, F32, L, (0, 8), 2, base=FAKE + (1 << 42))
    assert coco.raw_call("coco_looped_ag_einsum", b"mk,kn->mn", ctypes.byref(lhs), ctypes.byref(rhs),
                         ctypes.byref(out), None) == 0


def test_slice_validation(coco):
    F32, L, R, S = coco.F32, coco.LOCAL, coco.REPLICATED, coco.SLICED
    ins = mk(coco, F32, L, (24, 16), 4)
    # uneven slice: 24 rows do not split into... 24 % 4 == 0, so use 6 ranks of 4 rows is fine; 5 is not
    bad = mk(coco, F32, S, (24, 16), 5, slice_dim=0, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_reduce_scatter", ctypes.byref(mk(coco, F32, L, (24, 16), 5)), ctypes.byref(bad), None) == 2
    # slice_dim out of range
    bad = mk(coco, F32, S, (24, 16), 4, slice_dim=2, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_reduce_scatter", ctypes.byref(ins), ctypes.byref(bad), None) == 2
    # slice of the inner dimension that is not a multiple of 8 elements
    bad = mk(coco, F32, S, (24, 16), 4, slice_dim=1, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_reduce_scatter", ctypes.byref(ins), ctypes.byref(bad), None) == 5
    # wrong layouts
    good = mk(coco, F32, S, (24, 16), 4, slice_dim=0, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_reduce_scatter", ctypes.byref(good), ctypes.byref(good), None) == 4
    assert coco.raw_call("coco_allgather", ctypes.byref(ins), ctypes.byref(mk(coco, F32, R, (24, 16), 4)), None) == 4
    # global shape mismatch
    bad = mk(coco, F32, S, (48, 16), 4, slice_dim=0, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_reduce_scatter", ctypes.byref(ins), ctypes.byref(bad), None) == 2
    # reduce-scatter output overlapping an input
    bad = mk(coco, F32, S, (24, 16), 4, slice_dim=0, base=FAKE + 64)
    assert coco.raw_call("coco_reduce_scatter", ctypes.byref(ins), ctypes.byref(bad), None) == 6
    # rs-ag: scratch overlapping the output
    out = mk(coco, F32, R, (24, 16), 4, base=FAKE + (1 << 41))
    scr = mk(coco, F32, S, (24, 16), 4, slice_dim=0, base=FAKE + (1 << 41) + 64)
    assert coco.raw_call("coco_allreduce_rs_ag", ctypes.byref(ins), ctypes.byref(scr), ctypes.byref(out), None) == 6


def ein(coco, name, spec, lhs, rhs, out):
    return coco.raw_call(name, spec, ctypes.byref(lhs), ctypes.byref(rhs), ctypes.byref(out), None)


def test_einsum_validation(coco):
    B16, L, R, S = coco.BF16, coco.LOCAL, coco.REPLICATED, coco.SLICED
    lhs = mk(coco, B16, S, (64, 32), 4, slice_dim=0)
    rhs = mk(coco, B16, L, (32, 16), 4, base=FAKE + (1 << 40))
    out = mk(coco, B16, L, (64, 16), 4, base=FAKE + (1 << 41))
    A = "coco_looped_ag_einsum"
    assert ein(coco, A, b"mk,kn->nm", lhs, rhs, out) == 7            # unsupported spec
    assert ein(coco, A, b"bmk,bkn->bmn", lhs, rhs, out) == 2         # rank of operands vs spec
    assert ein(coco, A, b"mk,kn->mn", lhs, mk(coco, coco.F16, L, (32, 16), 4, base=FAKE + (1 << 40)), out) == 3
    assert ein(coco, A, b"mk,kn->mn", mk(coco, B16, L, (16, 32), 4), rhs, out) == 4   # nothing looped
    assert ein(coco, A, b"mk,kn->mn", lhs, mk(coco, B16, S, (32, 16), 4, slice_dim=0, base=FAKE + (1 << 40)), out) == 4
    assert ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, B16, R, (64, 16), 4, base=FAKE + (1 << 41))) == 4
    assert ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, B16, L, (16, 16), 4, base=FAKE + (1 << 41))) == 2
    assert ein(coco, A, b"mk,kn->mn", lhs, mk(coco, B16, L, (24, 16), 4, base=FAKE + (1 << 40)), out) == 2
    # output overlapping the local operand
    assert ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, B16, L, (64, 16), 4, base=FAKE + (1 << 40) + 16)) == 6
    RS = "coco_looped_einsum_rs"
    l2 = mk(coco, B16, S, (64, 32), 4, slice_dim=1)
    r2 = mk(coco, B16, S, (32, 16), 4, slice_dim=0, base=FAKE + (1 << 40))
    o2 = mk(coco, B16, S, (64, 16), 4, slice_dim=0, base=FAKE + (1 << 41))
    assert ein(coco, RS, b"mk,kn->mn", lhs, r2, o2) == 4     # lhs not sliced on k
    assert ein(coco, RS, b"mk,kn->mn", l2, r2, mk(coco, B16, L, (16, 16), 4, base=FAKE + (1 << 41))) == 4
    assert ein(coco, RS, b"mk,kn->mn", l2, r2, mk(coco, B16, S, (64, 24), 4, slice_dim=0, base=FAKE + (1 << 41))) == 2
    E = "coco_einsum"
    assert ein(coco, E, b"mk,kn->mn", lhs, rhs, out) == 4    # lhs sliced on m is not a local matmul
    assert ein(coco, E, b"mk,kn->mn", l2, r2, mk(coco, B16, R, (64, 16), 4, base=FAKE + (1 << 41))) == 4


def test_schedule_validation(coco):
    B16, L, S = coco.BF16, coco.LOCAL, coco.SLICED
    lhs = mk(coco, B16, S, (64, 32), 4, slice_dim=0)
    rhs = mk(coco, B16, L, (32, 16), 4, base=FAKE + (1 << 40))
    out = mk(coco, B16, L, (64, 16), 4, base=FAKE + (1 << 41))
    for name in ("coco_looped_ag_einsum_sched", "coco_looped_einsum_rs_sched"):
        for bad in (-1, 3, 99):
            assert coco.raw_call(name, b"mk,kn->mn", ctypes.byref(lhs), ctypes.byref(rhs), ctypes.byref(out),
                                 bad, None) == 10


def test_scattered_table_validation(coco):
    assert coco.coco_scattered_table_bytes([0], 4) == 64
    assert coco.coco_scattered_table_bytes([1024, 1025, 1], 8) == 64 + 12 * (1 + 2 + 1) * 8
    assert coco.coco_scattered_table_bytes([-1], 2) == 0
    lib = coco._lib
    numels = (ctypes.c_int64 * 2)(1000, 3000)
    plan = coco.CocoScatteredPlan()
    def build(ptrs, table=FAKE + (1 << 44), tbytes=1 << 20, dtype=coco.F16, nranks=2, nums=numels):
        arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
        return lib.coco_scattered_table_build(2, nums, dtype, nranks, arr, ctypes.c_void_p(table), tbytes,
                                              ctypes.byref(plan), None)
    good = [FAKE + i * (1 << 32) for i in range(4)]
    assert build(good, dtype=9) == 3
    assert build(good, nranks=0) == 2
    assert build([good[0], 0, good[2], good[3]]) == 1
    assert build([good[0] + 8] + good[1:]) == 5
    assert build(good, table=FAKE + (1 << 44) + 4) == 5
    assert build(good, tbytes=100) == 2
    assert build([good[0], good[0] + 64] + good[2:]) == 6          # overlapping tensors
    assert build(good, table=good[1] + 256) == 6                   # table inside a tensor
    big = (ctypes.c_int64 * 2)(1 << 32, 1)
    assert build(good, nums=big) == 2
    assert lib.coco_scattered_allreduce(None, ctypes.c_float(1.0), None) == 1
    p2 = coco.CocoScatteredPlan(None, 0, 2, coco.F16)
    assert lib.coco_scattered_allreduce(ctypes.byref(p2), ctypes.c_float(1.0), None) == 0  # nothing to do
    p3 = coco.CocoScatteredPlan(None, 5, 2, coco.F16)
    assert lib.coco_scattered_allreduce(ctypes.byref(p3), ctypes.c_float(1.0), None) == 1


def test_noalloc_rejects_overflowing_extents_before_any_cuda_call(coco):
    """Extents are range-checked one by one before they are multiplied: a shape whose product
    overflows 64 bits is refused with COCO_ERR_SHAPE like the caller-scratch entry point refuses it,
    not wrapped to an empty tensor."""
    F32, L, R, S = coco.F32, coco.LOCAL, coco.REPLICATED, coco.SLICED
    n = 8
    huge = (1 << 22, 1 << 21, 1 << 21)  # 2^64 elements: wraps to 0 in a plain int64 product
    for shape in [huge, (8, (1 << 40) + 8), (1 << 21, 1 << 20, 8)]:
        t = mk(coco, F32, L, shape, n)
        o = mk(coco, F32, R, shape, n, base=FAKE + (1 << 40))
        assert coco.raw_call("coco_allreduce_rs_ag_noalloc", ctypes.byref(t), ctypes.byref(o), None) == 2, shape
        sc = mk(coco, F32, S, shape, n, slice_dim=0, base=FAKE + (2 << 40))
        assert coco.raw_call("coco_allreduce_rs_ag", ctypes.byref(t), ctypes.byref(sc), ctypes.byref(o),
                             None) == 2, shape
    # structural errors still come first and an empty tensor is still a no-op
    t = mk(coco, F32, L, (0, 16), n)
    o = mk(coco, F32, R, (0, 16), n, base=FAKE + (1 << 40))
    assert coco.raw_call("coco_allreduce_rs_ag_noalloc", ctypes.byref(t), ctypes.byref(o), None) == 0
    assert coco.raw_call("coco_allreduce_rs_ag_noalloc", None, ctypes.byref(o), None) == 1


# ------------------------------------------- schedule query and cost model (host only)

def _traced_orders(kind, sched, n):
    """Per-rank orders read off the oracle's looped forms (shard IDs travel with the data there)."""
    import numpy as np
    import oracle
    ones = [np.ones((n, n)) for _ in range(n)]
    trace = []
    if kind == 0:
        if sched == 2:
            oracle.looped_allgather_einsum_bidirectional("mk,kn->mn", "lhs", "m", [np.ones((1, n))] * n,
                                                         [np.ones((n, n))] * n, trace)
        else:
            oracle.looped_allgather_einsum("mk,kn->mn", "lhs", "m", [np.ones((1, n))] * n, [np.ones((n, n))] * n,
                                           trace)
        return [[t[-1] for t in sorted(trace, key=lambda t: t[0]) if t[1] == r] for r in range(n)]
    if sched == 0:
        oracle.looped_einsum_reduce_scatter("mk,kn->mn", ones, ones, "m", trace)
        return [[q for (i, q, sid) in sorted(trace) if sid == r] for r in range(n)]
    if sched == 1:
        oracle.looped_einsum_reduce_scatter_unrolled("mk,kn->mn", ones, ones, "m", trace)
        return [[q for (i, q, c, sid) in sorted(trace) if sid == r and c == "A"] +
                [q for (i, q, c, sid) in sorted(trace) if sid == r and c == "B"] for r in range(n)]
    oracle.looped_einsum_reduce_scatter_bidirectional("mk,kn->mn", ones, ones, "m", trace)
    return [[q for (i, q, d, sid) in sorted(trace) if sid == r and d == "left"] +
            [q for (i, q, d, sid) in sorted(trace) if sid == r and d == "right"] + [r] for r in range(n)]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_shard_order_matches_the_oracles_schedules(coco, n):
    for kind in (0, 1):
        for sched in (0, 1, 2):
            want = _traced_orders(kind, sched, n)
            for r in range(n):
                got = coco.coco_shard_order(kind, sched, r, n)
                assert got == want[r], (kind, sched, n, r)
                assert sorted(got) == list(range(n))


def test_shard_order_validation(coco):
    NULL, SHAPE, VALUE = 1, 2, 10
    arr = (ctypes.c_int32 * 8)()
    assert coco.raw_call("coco_shard_order", 0, 0, 0, 8, None) == NULL
    assert coco.raw_call("coco_shard_order", 0, 0, 8, 8, arr) == SHAPE
    assert coco.raw_call("coco_shard_order", 0, 0, -1, 8, arr) == SHAPE
    assert coco.raw_call("coco_shard_order", 0, 0, 0, 0, arr) == SHAPE
    assert coco.raw_call("coco_shard_order", 0, 0, 0, 65, arr) == SHAPE
    assert coco.raw_call("coco_shard_order", 2, 0, 0, 8, arr) == VALUE
    assert coco.raw_call("coco_shard_order", 0, 3, 0, 8, arr) == VALUE


def test_loop_profitable_matches_the_oracle(coco):
    import numpy as np
    import oracle
    rng = np.random.default_rng(55)
    vals = [0.0, 0.25, 1.0, 2.0, 3.0, 4.0]
    cases = [(a, b, c, d) for a in vals for b in vals for c in vals for d in vals]
    cases += [tuple(rng.uniform(0, 10, 4)) for _ in range(2000)]
    for c in cases:
        assert coco.coco_loop_profitable(*c) == oracle.loop_profitable(*c), c


def test_loop_profitable_validation(coco):
    NULL, VALUE = 1, 10
    out = ctypes.c_int32(7)
    for bad in [(-1.0, 0, 0, 0), (0, -1e-9, 0, 0), (0, 0, float("nan"), 0), (0, 0, 0, float("inf"))]:
        assert coco.raw_call("coco_loop_profitable", *[ctypes.c_double(v) for v in bad],
                             ctypes.byref(out)) == VALUE
        assert out.value == 7  # untouched
    assert coco.raw_call("coco_loop_profitable", *[ctypes.c_double(1.0)] * 4, None) == \
        NULL


def test_plan_cache_keys_on_every_argument(coco):
    """A repeated call finds its plan; any changed pointer, shape, dtype, spec or schedule misses. Runs
    without a GPU: the keyed plans are entered after validation, and the status of a call that hits is
    the status of the call that made the plan (here the missing device's error, the same both times)."""
    B16, L, S = coco.BF16, coco.LOCAL, coco.SLICED
    coco.coco_plan_cache_clear()
    lhs = mk(coco, B16, S, (64, 32), 4, slice_dim=0)
    rhs = mk(coco, B16, L, (32, 16), 4, base=FAKE + (1 << 40))
    out = mk(coco, B16, L, (64, 16), 4, base=FAKE + (1 << 41))
    A = "coco_looped_ag_einsum"

    def delta(fn):
        h0, m0, _ = coco.coco_plan_cache_stats()
        st = fn()
        h1, m1, e1 = coco.coco_plan_cache_stats()
        return st, h1 - h0, m1 - m0, e1

    first, h, m, e = delta(lambda: ein(coco, A, b"mk,kn->mn", lhs, rhs, out))
    assert (h, m, e) == (0, 1, 1)
    again, h, m, e = delta(lambda: ein(coco, A, b"mk,kn->mn", lhs, rhs, out))
    assert (again, h, m, e) == (first, 1, 0, 1)
    # a changed pointer of one rank, a changed shape, another spec spelling, a schedule, an entry point
    moved = mk(coco, B16, L, (32, 16), 4, base=FAKE + (1 << 40))
    moved.ptr[3] = FAKE + (1 << 40) + 3 * (1 << 32) + 4096
    _, h, m, _ = delta(lambda: ein(coco, A, b"mk,kn->mn", lhs, moved, out))
    assert (h, m) == (0, 1)
    lhs2 = mk(coco, B16, S, (128, 32), 4, slice_dim=0)
    out2 = mk(coco, B16, L, (128, 16), 4, base=FAKE + (1 << 41))
    _, h, m, _ = delta(lambda: ein(coco, A, b"mk,kn->mn", lhs2, rhs, out2))
    assert (h, m) == (0, 1)
    _, h, m, _ = delta(lambda: ein(coco, A, b"mk, kn->mn", lhs, rhs, out))
    assert (h, m) == (0, 1)
    _, h, m, _ = delta(lambda: coco.raw_call("coco_looped_ag_einsum_sched", b"mk,kn->mn", ctypes.byref(lhs),
                                             ctypes.byref(rhs), ctypes.byref(out), 2, None))
    assert (h, m) == (0, 1)
    f16 = mk(coco, coco.F16, S, (64, 32), 4, slice_dim=0)
    _, h, m, _ = delta(lambda: ein(coco, A, b"mk,kn->mn", f16, mk(coco, coco.F16, L, (32, 16), 4,
                                                                  base=FAKE + (1 << 40)),
                                   mk(coco, coco.F16, L, (64, 16), 4, base=FAKE + (1 << 41))))
    assert (h, m) == (0, 1)
    # the original arguments still hit; a stream is not part of a plan
    _, h, m, _ = delta(lambda: coco.raw_call(A, b"mk,kn->mn", ctypes.byref(lhs), ctypes.byref(rhs),
                                             ctypes.byref(out), ctypes.c_void_p(0x1234)))
    assert (h, m) == (1, 0)
    # invalid calls are never entered
    _, _, _, e0 = delta(lambda: None)
    bad, h, m, e = delta(lambda: ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, B16, L, (16, 16), 4,
                                                                          base=FAKE + (1 << 41))))
    assert bad == 2 and e == e0
    coco.coco_plan_cache_clear()
    assert coco.coco_plan_cache_stats()[2] == 0


def test_plan_cache_under_concurrent_calls(coco):
    """Several host threads calling with the same and with different arguments at once: every call gets
    the status a single call gets, and the cache's counters account for every keyed call."""
    import threading
    B16, L, S = coco.BF16, coco.LOCAL, coco.SLICED
    coco.coco_plan_cache_clear()
    h0, m0, _ = coco.coco_plan_cache_stats()
    rhs = mk(coco, B16, L, (32, 16), 4, base=FAKE + (1 << 40))
    calls = []
    for t in range(8):
        lhs = mk(coco, B16, S, (64, 32), 4, slice_dim=0)
        out = mk(coco, B16, L, (64, 16), 4, base=FAKE + (1 << 41) + (t % 3) * (1 << 36))  # three distinct keys
        calls.append((lhs, out))
    want = ein(coco, "coco_looped_ag_einsum", b"mk,kn->mn", calls[0][0], rhs, calls[0][1])
    statuses, errors = [], []

    def worker(lhs, out):
        try:
            for _ in range(50):
                statuses.append(ein(coco, "coco_looped_ag_einsum", b"mk,kn->mn", lhs, rhs, out))
        except Exception as e:  # pragma: no cover
            errors.append(e)

    threads = [threading.Thread(target=worker, args=c) for c in calls]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors
    assert set(statuses) == {want} and len(statuses) == 400
    h1, m1, e1 = coco.coco_plan_cache_stats()
    assert (h1 - h0) + (m1 - m0) == 401 and e1 >= 3
    coco.coco_plan_cache_clear()


def test_einsum_accumulate_validation(coco):
    B16, L = coco.BF16, coco.LOCAL
    lhs = mk(coco, B16, L, (64, 32), 4)
    rhs = mk(coco, B16, L, (32, 16), 4, base=FAKE + (1 << 40))
    A = "coco_einsum_accumulate"
    assert ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, B16, L, (64, 16), 4, base=FAKE + (1 << 41))) == 3  # not fp32
    assert ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, coco.F32, coco.REPLICATED, (64, 16), 4,
                                                   base=FAKE + (1 << 41))) == 4
    assert ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, coco.F32, L, (64, 24), 4, base=FAKE + (1 << 41))) == 2
    assert ein(coco, A, b"mk,kn->mn", lhs, rhs, mk(coco, coco.F32, L, (64, 16), 4, base=FAKE + (1 << 40))) == 6
    empty_k = mk(coco, B16, L, (64, 0), 4)
    # zero contraction: nothing to add, no CUDA call
    assert ein(coco, A, b"mk,kn->mn", empty_k, mk(coco, B16, L, (0, 16), 4, base=FAKE + (1 << 40)),
               mk(coco, coco.F32, L, (64, 16), 4, base=FAKE + (1 << 41))) == 0
