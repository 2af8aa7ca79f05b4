"""The RS-AG entry point for callers that cannot allocate device memory.

Some callers may not call cudaMalloc once they are running (a latency-critical
loop where an allocation could stall or fail mid-step, or a plug-in inside an
application that owns all device memory). ``coco_allreduce_rs_ag_noalloc``
serves them: it takes only inputs and outputs and keeps the sliced
intermediate in a fixed 16 MiB array inside the library. These tests call it
through the C-ABI and compare it bit for bit with ``coco_allreduce_rs_ag``
given caller-owned scratch (both sum in fp32 in rank order), and with the
float64 oracle within the usual tolerance, on two calls in a row (the second
finds the first call's values in the shared array). They also check the size
limit at its exact edge, that a call leaves the device's free memory
unchanged, and that the one-time address look-up is refused on a stream that
is being captured.

This file is named so that pytest collects it last.
"""

import ctypes
import os
import subprocess
import sys

import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIMIT = 16 << 20  # bytes of the library's scratch array


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
        host = synth.per_rank(40 + call, 0, n * ngroups, shape, dtype, "uniform")
        ins = [t.cuda() for t in host]
        sl = (shape[0] // n,) + shape[1:]
        scratch = [torch.empty(sl, dtype=dtype, device="cuda") for _ in range(n * ngroups)]
        want = [torch.empty(shape, dtype=dtype, device="cuda") for _ in range(n * ngroups)]
        got = [torch.full(shape, float("nan"), dtype=dtype, device="cuda") for _ in range(n * ngroups)]
        coco.coco_allreduce_rs_ag(coco.local(ins, ngroups), coco.sliced(scratch, 0, ngroups),
                                  coco.replicated(want, ngroups))
        assert call_noalloc(coco, coco.local(ins, ngroups), coco.replicated(got, ngroups)) == 0
        torch.cuda.synchronize()
        for g in range(ngroups):
            ref = oracle.allreduce([synth.as_f64(x) for x in host[g * n:(g + 1) * n]])
            for r in range(n):
                q = g * n + r
                assert torch.equal(got[q], want[q]), f"call {call} group {g} rank {r}"
                assert_close(got[q], ref[r], dtype, f"call {call} group {g} rank {r} vs oracle")


def test_exact_limit_is_accepted_and_one_element_more_refused(coco):
    """8 ranks of fp32: 2^19 elements a slice fill the array exactly (8 slices of 2 MiB); one more
    element a slice rounds each slice up to the next 256 bytes and no longer fits."""
    n = 8
    numel = n * (LIMIT // n // 4)
    ins = [t.cuda() for t in synth.per_rank(44, 0, n, (numel,), torch.float32, "uniform")]
    want = [torch.empty(numel, device="cuda") for _ in range(n)]
    got = [torch.empty(numel, device="cuda") for _ in range(n)]
    scratch = [torch.empty(numel // n, device="cuda") for _ in range(n)]
    coco.coco_allreduce_rs_ag(coco.local(ins), coco.sliced(scratch, 0), coco.replicated(want))
    assert call_noalloc(coco, coco.local(ins), coco.replicated(got)) == 0
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        assert torch.equal(g, w)

    more = numel + n  # one element more in every slice
    big_in = [torch.zeros(more, device="cuda") for _ in range(n)]
    big_out = [torch.zeros(more, device="cuda") for _ in range(n)]
    before = coco.coco_kernel_launches()
    assert call_noalloc(coco, coco.local(big_in), coco.replicated(big_out)) == 7  # COCO_ERR_UNSUPPORTED
    assert coco.coco_kernel_launches() == before


def test_call_leaves_free_device_memory_unchanged(coco):
    n = 8
    shape = (1024, 256)
    ins = [t.cuda() for t in synth.per_rank(45, 0, n, shape, torch.bfloat16, "uniform")]
    got = [torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    assert call_noalloc(coco, coco.local(ins), coco.replicated(got)) == 0  # set-up done
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert call_noalloc(coco, coco.local(ins), coco.replicated(got)) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


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


_FIRST_CALL_UNDER_CAPTURE = r"""
import ctypes, sys, torch
sys.path.insert(0, sys.argv[1])
from collective_fusedallreduce_gb300 import coco
n = 4
ins = [torch.ones(64, device="cuda") for _ in range(n)]
outs = [torch.zeros(64, device="cuda") for _ in range(n)]
a, b = coco.local(ins).c(), coco.replicated(outs).c()
torch.cuda.synchronize()
s = torch.cuda.Stream()
with torch.cuda.stream(s):
    g = torch.cuda.CUDAGraph()
    g.capture_begin()
    st = coco.raw_call("coco_allreduce_rs_ag_noalloc", ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(s.cuda_stream))
    g.capture_end()
torch.cuda.synchronize()
assert st == 7, st  # the look-up is refused under capture; nothing was launched
st = coco.raw_call("coco_allreduce_rs_ag_noalloc", ctypes.byref(a), ctypes.byref(b), None)
torch.cuda.synchronize()
assert st == 0, st
assert all(bool((o == n).all()) for o in outs)
print("ok")
"""


def test_first_call_during_capture_is_refused_in_a_fresh_process(coco):
    """The address look-up happens on the first call in a process; on a stream being captured it is
    refused with COCO_ERR_UNSUPPORTED, and the same call outside capture then works."""
    p = subprocess.run([sys.executable, "-c", _FIRST_CALL_UNDER_CAPTURE, ROOT], capture_output=True, text=True,
                       timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip().endswith("ok")
