"""Full comparison at full size: every element of every rank's output of the
configurations the bench times, against the float64 oracle computed from the
same input values copied to the host.

The routine suite compares sampled rows at these sizes (the oracle's float64
GEMMs take minutes here); this module compares everything and is run once on
demand: ``COCO_FULL_ORACLE=1 python -m pytest tests/test_gpu_full_oracle.py -s``.
Each test prints the elements compared, the worst error scaled as in the
tolerance (|gpu - ref| / (|ref| + 1)) and the oracle's time on the host.
"""

import os
import time

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import TOL, f64

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(os.environ.get("COCO_FULL_ORACLE") != "1",
                       reason="the full-size float64 comparison runs on demand (COCO_FULL_ORACLE=1)"),
]

BF16, F16, F32 = torch.bfloat16, torch.float16, torch.float32


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


@pytest.fixture(scope="module")
def workloads(coco):
    from collective_fusedallreduce_gb300 import workloads as w
    return w


def cuda_gen(seed, shape, dtype, std=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.empty(shape, device="cuda").normal_(0.0, std, generator=g).to(dtype)


class Tally:
    """Worst scaled error over every compared element, and the oracle's host time."""

    def __init__(self, name, dtype):
        self.name, self.dtype = name, dtype
        self.worst, self.count, self.oracle_s = 0.0, 0, 0.0

    def oracle(self, fn, *args, **kw):
        t0 = time.perf_counter()
        r = fn(*args, **kw)
        self.oracle_s += time.perf_counter() - t0
        return r

    def compare(self, gpu, ref, what):
        g = f64(gpu)
        ref = np.asarray(ref, np.float64)
        assert g.shape == ref.shape, f"{what}: shape {g.shape} != {ref.shape}"
        assert np.isfinite(g).all(), f"{what}: non-finite output"
        err = np.abs(g - ref) / (np.abs(ref) + 1.0)
        w = float(err.max()) if err.size else 0.0
        self.worst = max(self.worst, w)
        self.count += err.size
        assert w <= TOL[self.dtype], f"{what}: max scaled error {w:.3e} > {TOL[self.dtype]}"

    def report(self):
        print(f"\n[full oracle] {self.name}: {self.count} elements, worst scaled error {self.worst:.3e} "
              f"(bar {TOL[self.dtype]}), oracle {self.oracle_s:.1f} s on {os.cpu_count()} host cores")


def _megatron_inputs(n=8, rows=8192, hidden=4096):
    ins = [cuda_gen(synth.seed_of(2, 0, r), (rows, hidden // n), F16) for r in range(n)]
    ws = [cuda_gen(synth.seed_of(2, 1, r), (hidden // n, hidden), F16, 0.02) for r in range(n)]
    bias = cuda_gen(synth.seed_of(2, 2), (hidden,), F16, 0.02)
    res = cuda_gen(synth.seed_of(2, 3), (rows, hidden), F16)
    return ins, ws, bias, res


def test_config2_megatron_tail_every_element(coco, workloads):
    """The unfused step (local MatMul, then the FusedAllReduce) and the fused MatMul + FusedAllReduce:
    all 8 replicas of [8192, 4096]."""
    n = 8
    ins, ws, bias, res = _megatron_inputs()
    _, out = workloads.megatron_attention_tail(ins, ws, bias, res, 0.1, 0)
    fused = [torch.empty_like(res) for _ in range(n)]
    coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(ins, 1), coco.sliced(ws, 0), bias,
                                     coco.replicated([res] * n), 0.1, 0, coco.replicated(fused))
    coco.coco_device_status()
    t = Tally("C2 Megatron tail (unfused step and fused MatMul, 8 replicas each)", F16)
    _, ref = t.oracle(oracle.megatron_attention_tail, [f64(a) for a in ins], [f64(w) for w in ws], f64(bias),
                      f64(res), 0.1, 0)
    for q in range(n):
        t.compare(out[q], ref, f"unfused replica {q}")
        t.compare(fused[q], ref, f"fused replica {q}")
    t.report()


def test_config3_case1_every_element(coco):
    n, m, k, nn = 8, 16384, 8192, 3072
    a = [cuda_gen(synth.seed_of(3, 0, s), (m // n, k), BF16, k ** -0.5) for s in range(n)]
    b = [cuda_gen(synth.seed_of(3, 1, r), (k, nn), BF16) for r in range(n)]
    out = [torch.empty((m, nn), dtype=BF16, device="cuda") for _ in range(n)]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(a, 0), coco.local(b), coco.local(out))
    coco.coco_device_status()
    t = Tally("C3 case 1 (8 ranks x [16384, 3072])", BF16)
    shards = [f64(x) for x in a]
    for r in range(n):
        ref = t.oracle(oracle.allgather_einsum, "mk,kn->mn", "lhs", "m", shards, [f64(b[r])])[0]
        t.compare(out[r], ref, f"rank {r}")
    t.report()


def test_config4a_case2_every_element(coco):
    n, m, k, nn = 8, 8192, 16384, 8192
    a = [cuda_gen(synth.seed_of(4, 0, s), (m, k // n), BF16) for s in range(n)]
    b = [cuda_gen(synth.seed_of(4, 1, r), (k, nn), BF16) for r in range(n)]
    out = [torch.empty((m, nn), dtype=F32, device="cuda") for _ in range(n)]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(a, 1), coco.local(b), coco.local(out))
    coco.coco_device_status()
    # bf16 inputs with fp32 accumulation and output: the 16-bit bar applies (as in the sampled test)
    t = Tally("C4a case 2 (8 ranks x [8192, 8192] fp32)", BF16)
    shards = [f64(x) for x in a]
    fp32_worst = 0.0
    for r in range(n):
        ref = t.oracle(oracle.allgather_einsum, "mk,kn->mn", "lhs", "k", shards, [f64(b[r])])[0]
        t.compare(out[r], ref, f"rank {r}")
        # outputs have magnitude ~sqrt(K) = 128; relative to that scale the fp32 sum is far tighter
        fp32_worst = max(fp32_worst, float((np.abs(f64(out[r]) - ref) / (np.abs(ref) + np.sqrt(k))).max()))
    t.report()
    print(f"[full oracle] C4a error relative to the output scale sqrt(K): {fp32_worst:.3e} (bar 1e-4)")
    assert fp32_worst < 1e-4


def test_config4b_case3_every_element(coco):
    n, bt, m, k, nn = 8, 64, 1024, 128, 1024
    ls = [cuda_gen(synth.seed_of(4, 2, s), (bt // n, m, k), BF16) for s in range(n)]
    rs = [cuda_gen(synth.seed_of(4, 3, r), (bt, k, nn), BF16) for r in range(n)]
    out = [torch.empty((bt, m, nn), dtype=BF16, device="cuda") for _ in range(n)]
    coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.sliced(ls, 0), coco.local(rs), coco.local(out))
    coco.coco_device_status()
    t = Tally("C4b case 3 (8 ranks x [64, 1024, 1024])", BF16)
    shards = [f64(x) for x in ls]
    for r in range(n):
        ref = t.oracle(oracle.allgather_einsum, "bmk,bkn->bmn", "lhs", "b", shards, [f64(rs[r])])[0]
        t.compare(out[r], ref, f"rank {r}")
    t.report()


def test_config5_mesh_every_element(coco, workloads):
    m_x, n_y, b, f, h = 2, 4, 8192, 8192, 32768
    keys = [(x, y) for x in range(m_x) for y in range(n_y)]
    xb = {k: cuda_gen(synth.seed_of(5, 0, i), (b // n_y, f // m_x), BF16) for i, k in enumerate(keys)}
    w1 = {k: cuda_gen(synth.seed_of(5, 1, i), (f // n_y, h // m_x), BF16, f ** -0.5) for i, k in enumerate(keys)}
    w2 = {k: cuda_gen(synth.seed_of(5, 2, i), (h // m_x, f // n_y), BF16, h ** -0.5) for i, k in enumerate(keys)}
    bufs = workloads.mlp_2d(xb, w1, w2, m_x, n_y)
    coco.coco_device_status()
    t = Tally("C5 2-D mesh MLP (8 devices x [2048, 4096])", BF16)
    ref = t.oracle(oracle.mlp_2d_forward, {k: f64(v) for k, v in xb.items()}, {k: f64(v) for k, v in w1.items()},
                   {k: f64(v) for k, v in w2.items()}, m_x, n_y)
    for k in keys:
        # h is rounded to bf16 between the einsums on the GPU; the oracle keeps float64
        t.compare(bufs["y"][k], ref[k], f"device {k}")
    t.report()
    del bufs
    torch.cuda.empty_cache()
