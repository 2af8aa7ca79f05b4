"""The plan cache of the einsum entry points on the GPU: a repeated call reuses
its plan and gives the same bits, a call that differs in one pointer gets its
own plan and writes where it is told, and a cached call costs less host time
than planning afresh."""

import ctypes
import time

import pytest
import torch

from collective_fusedallreduce_gb300 import coco, synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _case1(n=8, m=256, k=512, nn=512, seed=401):
    shards = [t.to(DEV) for t in synth.per_rank(seed, 0, n, (m, k), torch.bfloat16, std=k ** -0.5)]
    rhs = [t.to(DEV) for t in synth.per_rank(seed, 1, n, (k, nn), torch.bfloat16)]
    return shards, rhs


def test_repeated_calls_hit_and_give_the_same_bits():
    n = 8
    shards, rhs = _case1()
    outs = [[torch.full((n * 256, 512), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
            for _ in range(3)]
    coco.coco_plan_cache_clear()
    h0, m0, _ = coco.coco_plan_cache_stats()
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(shards, 0), coco.local(rhs), coco.local(outs[0]))
    for o1, o0 in zip(outs[1], outs[0]):
        o1.copy_(o0)  # the first (planned) call's result
        o0.fill_(float("nan"))
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(shards, 0), coco.local(rhs), coco.local(outs[0]))
    h1, m1, e1 = coco.coco_plan_cache_stats()
    assert (h1 - h0, m1 - m0, e1) == (1, 1, 1)
    # one rank's output elsewhere: a new plan, and the result lands there
    moved = list(outs[0])
    moved[5] = outs[2][5]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(shards, 0), coco.local(rhs), coco.local(moved))
    h2, m2, _ = coco.coco_plan_cache_stats()
    assert (h2 - h1, m2 - m1) == (0, 1)
    coco.coco_device_status()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    assert torch.equal(outs[2][5], outs[0][5])
    assert torch.isnan(outs[2][4].float()).all()  # untouched


def test_fused_matmul_plan_keys_on_its_scalars():
    n, rows, hid = 4, 256, 512
    ins = [t.to(DEV) for t in synth.per_rank(402, 0, n, (rows, hid // n), torch.float16)]
    ws = [t.to(DEV) for t in synth.per_rank(402, 1, n, (hid // n, hid), torch.float16, std=0.02)]
    bias = synth.tensor(synth.seed_of(402, 2), (hid,), torch.float16, std=0.02).to(DEV)
    res = synth.tensor(synth.seed_of(402, 3), (rows, hid), torch.float16).to(DEV)
    a = [torch.empty((rows, hid), dtype=torch.float16, device=DEV) for _ in range(n)]
    b = [torch.empty_like(x) for x in a]
    c = [torch.empty_like(x) for x in a]
    args = (coco.sliced(ins, 1), coco.sliced(ws, 0), bias, coco.replicated([res] * n))
    coco.coco_plan_cache_clear()
    coco.coco_matmul_fused_allreduce("mk,kn->mn", *args, 0.1, 7, coco.replicated(a))
    coco.coco_matmul_fused_allreduce("mk,kn->mn", *args, 0.1, 8, coco.replicated(b))  # another seed
    _, m, _ = coco.coco_plan_cache_stats()
    coco.coco_matmul_fused_allreduce("mk,kn->mn", *args, 0.1, 7, coco.replicated(c))
    coco.coco_device_status()
    assert not torch.equal(a[0], b[0])  # the seed is part of the plan: a different mask
    ref = [torch.empty_like(x) for x in a]
    coco.coco_plan_cache_clear()
    coco.coco_matmul_fused_allreduce("mk,kn->mn", *args, 0.1, 7, coco.replicated(ref))
    coco.coco_device_status()
    assert torch.equal(c[0], ref[0]) and torch.equal(a[0], ref[0])


def test_cached_calls_cost_less_host_time():
    n = 8
    shards, rhs = _case1()
    out = [torch.empty((n * 256, 512), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    L, R, O = coco.sliced(shards, 0).c(), coco.local(rhs).c(), coco.local(out).c()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        t0 = time.perf_counter()
        st = coco.raw_call("coco_looped_ag_einsum", b"mk,kn->mn", ctypes.byref(L), ctypes.byref(R),
                           ctypes.byref(O), s)
        dt = time.perf_counter() - t0
        assert st == 0
        return dt

    fresh, cached = [], []
    for _ in range(30):
        coco.coco_plan_cache_clear()
        fresh.append(call())
        cached.append(call())
        torch.cuda.synchronize()
    fresh.sort()
    cached.sort()
    assert cached[15] < fresh[15], (cached[15], fresh[15])
