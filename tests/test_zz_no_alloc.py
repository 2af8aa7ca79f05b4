"""The RS-AG entry point for callers that cannot allocate device memory.

Some callers may not call cudaMalloc once they are running (a latency-critical
loop where an allocation could stall or fail mid-step, or a plug-in inside an
application that owns all device memory). ``coco_allreduce_rs_ag_noalloc``
serves them: it takes only inputs and outputs and keeps the sliced
intermediate in a fixed array inside the library. These tests call it through
the C-ABI and compare it with ``coco_allreduce_rs_ag`` given caller-owned
scratch, on two calls in a row (the second reuses the array the first left
behind), and check that an oversized request is refused.

This file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


def call_noalloc(coco, inp, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return coco.raw_call("coco_allreduce_rs_ag_noalloc", ctypes.byref(inp.c()), ctypes.byref(out.c()), stream)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_matches_caller_scratch_version_on_two_calls(coco, dtype):
    n = 8
    # two calls in a row with different shapes and data: the second call finds
    # the first call's values in the shared array
    for call, (shape, ngroups) in enumerate([((64, 96), 1), ((40, 3, 16), 2)]):
        ins = [t.cuda() for t in synth.per_rank(40 + call, 0, n * ngroups, shape, dtype, "uniform")]
        sl = (shape[0] // n,) + shape[1:]
        scratch = [torch.empty(sl, dtype=dtype, device="cuda") for _ in range(n * ngroups)]
        want = [torch.empty(shape, dtype=dtype, device="cuda") for _ in range(n * ngroups)]
        got = [torch.full(shape, float("nan"), dtype=dtype, device="cuda") for _ in range(n * ngroups)]
        coco.coco_allreduce_rs_ag(coco.local(ins, ngroups), coco.sliced(scratch, 0, ngroups),
                                  coco.replicated(want, ngroups))
        assert call_noalloc(coco, coco.local(ins, ngroups), coco.replicated(got, ngroups)) == 0
        torch.cuda.synchronize()
        for q, (g, w) in enumerate(zip(got, want)):
            assert_close(g, f64(w), dtype, f"call {call} rank {q}")


def test_oversized_request_is_refused_before_any_launch(coco):
    n = 8
    t = coco.CocoTensor()
    t.dtype, t.layout, t.ndim, t.slice_dim = coco.F32, coco.LOCAL, 2, -1
    t.shape[0], t.shape[1] = 8, 1 << 20  # 32 MiB of fp32 scratch > the 16 MiB array
    t.nranks, t.ngroups = n, 1
    for i in range(n):
        t.ptr[i] = 0x7F0000000000 + i * (1 << 32)
    o = coco.CocoTensor.from_buffer_copy(t)
    o.layout = coco.REPLICATED
    for i in range(n):
        o.ptr[i] = 0x7E0000000000 + i * (1 << 32)
    before = coco.coco_kernel_launches()
    assert coco.raw_call("coco_allreduce_rs_ag_noalloc", ctypes.byref(t), ctypes.byref(o), None) == 7
    assert coco.coco_kernel_launches() == before
