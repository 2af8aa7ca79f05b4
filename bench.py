#!/usr/bin/env python
"""Benchmark of the fused / looped collectives on one GB300 (or N replicas).

A step is one pass of the hot path over one batch of synthetic input, all N
logical ranks on this GPU. The default (headline) workload is the Megatron
self-attention output projection of [CoCoNet] Fig. 3: 8 ranks, fp16,
in[8,1024,4096] sliced on its last dimension, w[4096,4096] sliced on its
first, bias[4096], dropout p=0.1 and a replicated residual[8,1024,4096], with
the per-rank MatMul fused into the FusedAllReduce (one tensor-core kernel; no
partial is stored). After it, in the same process, every other configuration
is timed and reported as a sub-record under ``configs``: the unfused chain of
the same tail (``c2``: local MatMul, then FusedAllReduce), the looped
AllGather-Einsum cases 1/2/3 (``c3``, ``c4a``, ``c4b``), the 2-D mesh MLP
(``c5``), the RS-AG split AllReduce and the direct AllReduce of 1 GiB fp32 x 8
(``c5b``, ``c5d``) and the scattered-tensor AllReduce (``scatter``).
``--workload`` selects another headline (then no sub-records unless
``--configs`` names them).

``value`` is the step's throughput as a percentage of one GB300's roofline:
100 * ideal step time / measured step time, the ideal being the workload's own
roofline at the peaks of MEASURED_PEAKS.json (HBM copy GB/s and cuBLAS bf16
TFLOP/s burst; fp16 runs at the bf16 rate): for the fused tail max(MatMul
FLOPs, minimal traffic), for a chain of kernels the sum of each kernel's
ideal. Under torchrun every rank runs an independent replica on its own GPU
(weak scaling) and ``value`` sums the replicas' throughput.

``--impl reference`` times the CPU oracle (plain float64 NumPy) on host cores
on a bounded sample of the same workload, in the same unit.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "FusedAllReduce GB/s & looped CollectiveEinsum TFLOP/s, % of 1×GB300 roofline"
UNIT = "% of 1xGB300 roofline"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
MiB = 1 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK)


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi clock / throttle samples of this GPU while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index, period_ms=20):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device_index)
        self.cmd = ["nvidia-smi", "-i", ident, "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", str(period_ms)]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) != len(self.FIELDS):
                continue
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except ValueError:
                continue
            for name, v in zip(names, r[3:]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workloads


def gen(dev, seed, shape, dtype, std=1.0, kind="normal"):
    """Seeded synthetic device tensor (torch's CUDA generator; values only)."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.empty(shape, dtype=torch.float32, device=dev)
    if kind == "normal":
        x.normal_(0.0, std, generator=g)
    else:
        x.uniform_(-1.0, 1.0, generator=g)
    return x.to(dtype)


class Workload:
    """A step of the hot path: inputs, launches, algorithmic work and an oracle sample."""

    name = ""
    config = {}
    dtype = "f16"

    def kernels(self):
        """[(name, bound, units per launch, launches per step)], bound "hbm" (bytes) or "tensor" (flops)."""
        raise NotImplementedError

    def timed(self):
        """The segments timed with events inside a step (default: one per kernel)."""
        return self.kernels()

    def ideal_seconds(self, peaks):
        t = 0.0
        for _, bound, units, launches in self.kernels():
            t += launches * (units / (peaks["hbm_gbs"] * 1e9) if bound == "hbm" else units / (peaks["bf16_tflops"] * 1e12))
        return t

    def step(self, stream, marks=None):
        raise NotImplementedError

    def host_inputs(self):
        """[(device tensor, pinned host copy)] re-uploaded every e2e step, and the result tensor read back."""
        raise NotImplementedError

    def rebind(self, key):
        """Called after the input tensors were pointed at buffer set ``key``: rebuild any state that holds
        their addresses (none by default: every call reads the tensors' current pointers)."""

    def oracle_sample(self, rows):
        """Runs the oracle on a sample; returns the sample's fraction of the step's work."""
        raise NotImplementedError

    def sample_unit(self):
        return "rows"

    def full_sample(self):
        return 1


class MegatronTail(Workload):
    """[CoCoNet] Fig. 3: layer_r = in_r @ w_r (8 ranks, fp16), then FusedAllReduce."""

    name = "megatron_attention_tail"
    dtype = "f16"

    def __init__(self, dev, n=8, rows=8192, hidden=4096, p=0.1, seed=0, cfg=2):
        from collective_fusedallreduce_gb300 import synth
        self.n, self.rows, self.h, self.ks, self.p, self.seed = n, rows, hidden, hidden // n, p, seed
        f16 = torch.float16
        self.inp = [gen(dev, synth.seed_of(cfg, 0, r), (rows, self.ks), f16) for r in range(n)]
        self.w = [gen(dev, synth.seed_of(cfg, 1, r), (self.ks, hidden), f16, 0.02) for r in range(n)]
        self.bias = gen(dev, synth.seed_of(cfg, 2), (hidden,), f16, 0.02)
        self.res = gen(dev, synth.seed_of(cfg, 3), (rows, hidden), f16)
        self.layer = [torch.empty((rows, hidden), dtype=f16, device=dev) for _ in range(n)]
        self.out = [torch.empty((rows, hidden), dtype=f16, device=dev) for _ in range(n)]
        self.config = {"workload": "Megatron self-attention output projection (CoCoNet Fig. 3): N=8 ranks fp16, "
                                   "in[8,1024,4096] sliced dim 2, w[4096,4096] sliced dim 0, local MatMul -> "
                                   "FusedAllReduce + bias[4096] + dropout p=0.1 + residual[8,1024,4096]",
                       "ranks": n, "in_per_rank": [rows, self.ks], "w_per_rank": [self.ks, hidden],
                       "outputs": "8 distinct replicated copies",
                       "l2": "no flush: every step streams ~1.2 GB (> 126 MB L2)",
                       "inputs": "synthetic N(0,1) activations/residual, N(0,0.02) weights/bias"}

    def kernels(self):
        n, rows, h, ks = self.n, self.rows, self.h, self.ks
        flops = 2.0 * n * rows * ks * h
        far_bytes = (n * rows * h + rows * h + n * rows * h) * 2 + h * 2
        return [("k_gemm_tc (local MatMul, 8 ranks)", "tensor", flops, 1),
                ("k_fused_allreduce (8 ranks, bias+dropout+residual)", "hbm", far_bytes, 1)]

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        n = self.n
        if marks:
            marks[0].record(stream)
        coco.coco_einsum("mk,kn->mn", coco.sliced(self.inp, 1), coco.sliced(self.w, 0), coco.local(self.layer), stream)
        if marks:
            marks[1].record(stream)
        coco.coco_fused_allreduce(coco.local(self.layer), self.bias, coco.replicated([self.res] * n), self.p,
                                  self.seed, coco.replicated(self.out), stream)
        if marks:
            marks[2].record(stream)

    def host_inputs(self):
        ins = [(t, t.cpu().pin_memory()) for t in self.inp + self.w + [self.bias, self.res]]
        return ins, self.out[0]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        rng = np.random.default_rng(rows)
        sel = np.sort(rng.choice(self.rows, rows, replace=False))
        # host copies of the sampled inputs, taken before the clock starts
        ins = [synth.as_f64(x[sel]) for x in self.inp]
        ws = [synth.as_f64(x) for x in self.w]
        b = synth.as_f64(self.bias)
        res = synth.as_f64(self.res[sel])
        idx = sel[:, None].astype(np.uint64) * np.uint64(self.h) + np.arange(self.h, dtype=np.uint64)[None, :]
        t0 = time.perf_counter()
        layers = [oracle.einsum("mk,kn->mn", a, w) for a, w in zip(ins, ws)]
        oracle.fused_allreduce(layers, b, res, self.p, self.seed, index=idx)
        dt = time.perf_counter() - t0
        return dt, rows / self.rows

    def full_sample(self):
        return self.rows


class MegatronTailOverlap(MegatronTail):
    """[CoCoNet] §5.3 Overlap: the same Fig. 3 tail with the rows cut into chunks; the FusedAllReduce of
    chunk c (a second stream) runs while the MatMul computes chunk c+1. Stream order only: every
    FusedAllReduce waits for its chunk's MatMul through an event, nothing spins on the device.
    Dropout indices continue across chunks (coco_fused_allreduce_at), so the outputs equal the
    unchunked step's bit for bit. Rated against the whole step's own roofline, max(MatMul FLOPs at
    the tensor peak, MatMul + FusedAllReduce bytes at the HBM peak)."""

    name = "megatron_attention_tail_overlap"

    def __init__(self, dev, chunks=4, **kw):
        super().__init__(dev, **kw)
        self.chunks = chunks
        self.side = torch.cuda.Stream(device=dev)
        self.config = dict(self.config)
        self.config["workload"] = self.config["workload"].replace(
            "local MatMul -> FusedAllReduce",
            f"local MatMul overlapped with FusedAllReduce in {chunks} row chunks (two streams)")
        self.config["chunks"] = chunks

    def gemm_bytes(self):
        n, rows, h, ks = self.n, self.rows, self.h, self.ks
        return (n * rows * ks + n * ks * h + n * rows * h) * 2

    def timed(self):
        flops = self.kernels()[0][2]
        byts = self.kernels()[1][2] + self.gemm_bytes()
        return [(f"MatMul || FusedAllReduce in {self.chunks} chunks (step bytes)", "hbm", byts, 1)]

    def ideal_seconds(self, peaks):
        flops = self.kernels()[0][2]
        byts = self.kernels()[1][2] + self.gemm_bytes()
        return max(flops / (peaks["bf16_tflops"] * 1e12), byts / (peaks["hbm_gbs"] * 1e9))

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import workloads
        if marks:
            marks[0].record(stream)
        workloads.megatron_attention_tail_overlap(self.inp, self.w, self.bias, self.res, self.p, self.seed,
                                                  self.chunks, self.layer, self.out, stream, self.side)
        if marks:
            marks[1].record(stream)


class MegatronTailFused(MegatronTail):
    """The same Fig. 3 tail with the MatMul fused into the FusedAllReduce: one
    tensor-core kernel sums the 8 ranks' K-slices in TMEM and applies bias,
    dropout and residual in its epilogue; no per-rank partial is stored."""

    name = "megatron_attention_tail_fused"

    def __init__(self, dev, **kw):
        super().__init__(dev, **kw)
        self.config = dict(self.config)
        self.config["workload"] = self.config["workload"].replace(
            "local MatMul -> FusedAllReduce", "MatMul fused into FusedAllReduce (one kernel, no partials)")

    def kernels(self):
        n, rows, h, ks = self.n, self.rows, self.h, self.ks
        flops = 2.0 * n * rows * ks * h
        return [("k_gemm_tc<fused allreduce> (8 ranks' K-slices, bias+dropout+residual, 8 replicas)", "tensor",
                 flops, 1)]

    def min_bytes(self):
        n, rows, h, ks = self.n, self.rows, self.h, self.ks
        return (n * rows * ks + n * ks * h + rows * h + h + n * rows * h) * 2

    def ideal_seconds(self, peaks):
        # the fused computation's own roofline: max of its compute and its minimal traffic
        flops = self.kernels()[0][2]
        return max(flops / (peaks["bf16_tflops"] * 1e12), self.min_bytes() / (peaks["hbm_gbs"] * 1e9))

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        if marks:
            marks[0].record(stream)
        coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(self.inp, 1), coco.sliced(self.w, 0), self.bias,
                                         coco.replicated([self.res] * self.n), self.p, self.seed,
                                         coco.replicated(self.out), stream)
        if marks:
            marks[1].record(stream)


class LoopedCase1(Workload):
    """Looped AllGather-Einsum case 1: A[16384,8192] sliced on rows over 8 ranks, B_r[8192,3072] local, bf16."""

    name = "looped_ag_einsum_case1"
    dtype = "bf16"

    def __init__(self, dev, n=8, m=16384, k=8192, nn=3072, cfg=3):
        from collective_fusedallreduce_gb300 import synth
        bf = torch.bfloat16
        self.n, self.m, self.k, self.nn = n, m, k, nn
        self.a = [gen(dev, synth.seed_of(cfg, 0, s), (m // n, k), bf, k ** -0.5) for s in range(n)]
        self.b = [gen(dev, synth.seed_of(cfg, 1, r), (k, nn), bf) for r in range(n)]
        self.out = [torch.empty((m, nn), dtype=bf, device=dev) for _ in range(n)]
        self.config = {"workload": "Looped AllGather-Einsum case 1: N=8 bf16, A[16384,8192] sliced on rows, "
                                   "B_r[8192,3072] local, out_r[16384,3072] by DynamicUpdateSlice", "ranks": n,
                       "l2": "no flush: each step writes 768 MiB of output (> 126 MB L2)"}

    def kernels(self):
        return [("k_gemm_tc (case 1, 8 ranks x 8 steps)", "tensor", 2.0 * self.n * self.m * self.k * self.nn, 1)]

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        if marks:
            marks[0].record(stream)
        coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(self.a, 0), coco.local(self.b), coco.local(self.out), stream)
        if marks:
            marks[1].record(stream)

    def host_inputs(self):
        return [(t, t.cpu().pin_memory()) for t in self.a + self.b], self.out[0]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        per = max(1, rows // self.n)
        sel = np.sort(np.random.default_rng(rows).choice(self.m // self.n, per, replace=False))
        shards = [synth.as_f64(a[sel]) for a in self.a]
        bs = [synth.as_f64(b) for b in self.b]
        t0 = time.perf_counter()
        oracle.allgather_einsum("mk,kn->mn", "lhs", "m", shards, bs)
        return time.perf_counter() - t0, per * self.n / self.m

    def full_sample(self):
        return self.m


class LoopedCase2(Workload):
    """Looped AllGather-Einsum case 2: LHS[8192,16384] sliced on K, RHS_r[16384,8192] local, fp32 out."""

    name = "looped_ag_einsum_case2"
    dtype = "bf16"

    def __init__(self, dev, n=8, m=8192, k=16384, nn=8192, cfg=4):
        from collective_fusedallreduce_gb300 import synth
        bf = torch.bfloat16
        self.n, self.m, self.k, self.nn = n, m, k, nn
        self.a = [gen(dev, synth.seed_of(cfg, 0, s), (m, k // n), bf) for s in range(n)]
        self.b = [gen(dev, synth.seed_of(cfg, 1, r), (k, nn), bf) for r in range(n)]
        self.out = [torch.empty((m, nn), dtype=torch.float32, device=dev) for _ in range(n)]
        self.config = {"workload": "Looped AllGather-Einsum case 2: N=8 bf16, LHS[8192,16384] sliced on K, "
                                   "RHS_r[16384,8192] DynamicSliced along K, fp32 Addition in TMEM", "ranks": n,
                       "l2": "no flush: each step writes 2 GiB of output"}

    def kernels(self):
        return [("k_gemm_tc (case 2, 8 ranks, 8 K-segments)", "tensor", 2.0 * self.n * self.m * self.k * self.nn, 1)]

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        if marks:
            marks[0].record(stream)
        coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(self.a, 1), coco.local(self.b), coco.local(self.out), stream)
        if marks:
            marks[1].record(stream)

    def host_inputs(self):
        return [(t, t.cpu().pin_memory()) for t in self.a + self.b], self.out[0]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        sel = np.sort(np.random.default_rng(rows).choice(self.m, rows, replace=False))
        shards = [synth.as_f64(a[sel]) for a in self.a]
        bs = [synth.as_f64(b) for b in self.b]
        t0 = time.perf_counter()
        oracle.allgather_einsum("mk,kn->mn", "lhs", "k", shards, bs)
        return time.perf_counter() - t0, rows / self.m

    def full_sample(self):
        return self.m


class LoopedCase3(Workload):
    """Looped AllGather-Einsum case 3: L[64,1024,128] sliced on batch, R_r[64,128,1024], bf16."""

    name = "looped_ag_einsum_case3"
    dtype = "bf16"

    def __init__(self, dev, n=8, b=64, m=1024, k=128, nn=1024, cfg=4):
        from collective_fusedallreduce_gb300 import synth
        bf = torch.bfloat16
        self.n, self.b, self.m, self.k, self.nn = n, b, m, k, nn
        self.l = [gen(dev, synth.seed_of(cfg, 2, s), (b // n, m, k), bf) for s in range(n)]
        self.r = [gen(dev, synth.seed_of(cfg, 3, r), (b, k, nn), bf) for r in range(n)]
        self.out = [torch.empty((b, m, nn), dtype=bf, device=dev) for _ in range(n)]
        self.config = {"workload": "Looped AllGather-Einsum case 3: N=8 bf16, L[64,1024,128] sliced on batch, "
                                   "R_r[64,128,1024] DynamicSliced on batch, out_r[64,1024,1024] by "
                                   "DynamicUpdateSlice on batch", "ranks": n,
                       "l2": "no flush: each step writes 1 GiB of output"}

    def kernels(self):
        n, b, m, k, nn = self.n, self.b, self.m, self.k, self.nn
        byts = (b * m * k + n * b * k * nn + n * b * m * nn) * 2
        return [("k_gemm_tc (case 3, 8 ranks x 8 steps)", "hbm", byts, 1)]

    def flops(self):
        return 2.0 * self.n * self.b * self.m * self.k * self.nn

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        if marks:
            marks[0].record(stream)
        coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.sliced(self.l, 0), coco.local(self.r), coco.local(self.out),
                                   stream)
        if marks:
            marks[1].record(stream)

    def host_inputs(self):
        return [(t, t.cpu().pin_memory()) for t in self.l + self.r], self.out[0]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        per = max(1, rows // self.n)
        ls = [synth.as_f64(x[:, :per]) for x in self.l]
        rs = [synth.as_f64(x) for x in self.r]
        t0 = time.perf_counter()
        oracle.allgather_einsum("bmk,bkn->bmn", "lhs", "b", ls, rs)
        return time.perf_counter() - t0, per / self.m

    def full_sample(self):
        return self.m * self.n


class Mesh2D(Workload):
    """[Decomp] §2.2 Fig. 3 MLP on a [2, 4] mesh, bf16, B=8192, F=8192, H=32768."""

    name = "mlp_2d_mesh"
    dtype = "bf16"

    def __init__(self, dev, m_x=2, n_y=4, b=8192, f=8192, h=32768, cfg=5):
        from collective_fusedallreduce_gb300 import synth
        bf = torch.bfloat16
        self.mx, self.ny, self.b, self.f, self.h = m_x, n_y, b, f, h
        keys = [(x, y) for x in range(m_x) for y in range(n_y)]
        d = {k: x * n_y + y for k, (x, y) in zip(keys, keys)}
        self.x = {k: gen(dev, synth.seed_of(cfg, 0, d[k]), (b // n_y, f // m_x), bf) for k in keys}
        self.w1 = {k: gen(dev, synth.seed_of(cfg, 1, d[k]), (f // n_y, h // m_x), bf, f ** -0.5) for k in keys}
        self.w2 = {k: gen(dev, synth.seed_of(cfg, 2, d[k]), (h // m_x, f // n_y), bf, h ** -0.5) for k in keys}
        self.bufs = None
        from collective_fusedallreduce_gb300 import workloads
        self.bufs = workloads.mlp_2d(self.x, self.w1, self.w2, m_x, n_y)  # allocates buffers
        self.side = torch.cuda.Stream(device=dev)  # the AllGather of W2 runs beside the first einsum
        self.config = {"workload": "2-D mesh [M=2,N=4] MLP (Decomp Fig. 3), bf16, B=8192 F=8192 H=32768: AG X "
                                   "along x, looped AG-einsum of W1 along y, AG W2 along y, looped einsum-RS along x",
                       "devices": m_x * n_y, "l2": "no flush: each step moves > 4 GB"}

    def kernels(self):
        mx, ny, b, f, h = self.mx, self.ny, self.b, self.f, self.h
        dev = mx * ny
        ein = 2.0 * dev * (b // ny) * f * (h // mx)
        ag_x = dev * (b // ny) * (f // mx) * 2 + dev * (b // ny) * f * 2
        ag_w2 = dev * (h // mx) * (f // ny) * 2 + dev * (h // mx) * f * 2
        return [("k_gemm_tc (looped AG-einsum of W1, case 2)", "tensor", ein, 1),
                ("k_gemm_tc (looped einsum-RS along x)", "tensor", ein, 1),
                ("k_allgather (X along x)", "hbm", ag_x, 1),
                ("k_allgather (W2 along y)", "hbm", ag_w2, 1)]

    def timed(self):
        ein = sum(k[2] for k in self.kernels() if k[1] == "tensor")
        return [("2-D mesh MLP step (2 looped einsums + 2 all-gathers), einsum FLOPs", "tensor", ein, 1)]

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import workloads
        if marks:
            marks[0].record(stream)
        workloads.mlp_2d(self.x, self.w1, self.w2, self.mx, self.ny, self.bufs, stream, self.side)
        if marks:
            marks[1].record(stream)

    def host_inputs(self):
        ts = list(self.x.values()) + list(self.w1.values()) + list(self.w2.values())
        return [(t, t.cpu().pin_memory()) for t in ts], self.bufs["y"][(0, 0)]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        per = max(1, rows // self.ny)
        xs = {k: synth.as_f64(v[:per]) for k, v in self.x.items()}
        w1 = {k: synth.as_f64(v) for k, v in self.w1.items()}
        w2 = {k: synth.as_f64(v) for k, v in self.w2.items()}
        t0 = time.perf_counter()
        oracle.mlp_2d_forward(xs, w1, w2, self.mx, self.ny)
        return time.perf_counter() - t0, per / (self.b // self.ny)

    def full_sample(self):
        return self.b


class RsAg(Workload):
    """AllReduce Split RS-AG of a 1 GiB fp32 tensor over 8 ranks."""

    name = "allreduce_split_rs_ag"
    dtype = "f32"

    def __init__(self, dev, n=8, numel=1 << 28, cfg=5, small=False):
        from collective_fusedallreduce_gb300 import synth
        numel = numel >> 3 if small else numel
        self.n, self.numel = n, numel
        self.inp = [gen(dev, synth.seed_of(cfg, 5, r), (numel,), torch.float32, kind="uniform") for r in range(n)]
        self.scratch = [torch.empty(numel // n, device=dev) for _ in range(n)]
        self.out = [torch.empty(numel, device=dev) for _ in range(n)]
        self.config = {"workload": f"AllReduce split RS-AG, N=8 fp32, {numel} elements ({numel * 4 >> 20} MiB) per "
                                   f"rank, 8 distinct outputs", "ranks": n,
                       "l2": f"no flush: each step moves {18 * numel * 4 >> 30} GiB"}

    def kernels(self):
        b = self.numel * 4
        return [("k_reduce_scatter", "hbm", self.n * b + b, 1), ("k_allgather", "hbm", b + self.n * b, 1)]

    def timed(self):
        return [("k_reduce_scatter + k_allgather (one coco_allreduce_rs_ag call)", "hbm",
                 sum(k[2] for k in self.kernels()), 1)]

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        if marks:
            marks[0].record(stream)
        coco.coco_allreduce_rs_ag(coco.local(self.inp), coco.sliced(self.scratch, 0), coco.replicated(self.out), stream)
        if marks:
            marks[1].record(stream)

    def host_inputs(self):
        return [(t, t.cpu().pin_memory()) for t in self.inp], self.out[0]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        cnt = rows * 4096
        xs = [synth.as_f64(x[:cnt]) for x in self.inp]
        t0 = time.perf_counter()
        oracle.allreduce_split_rs_ag(xs, 0)
        return time.perf_counter() - t0, cnt / self.numel

    def full_sample(self):
        return self.numel // 4096


class AllReduceDirect(RsAg):
    """The direct AllReduce of the same 1 GiB fp32 tensor over 8 ranks (one N-way reduction kernel,
    no scratch), for comparison with the RS-AG split; bit-identical to it."""

    name = "allreduce_direct"

    def __init__(self, dev, n=8, numel=1 << 28, cfg=5, small=False):
        super().__init__(dev, n, numel, cfg, small)
        self.scratch = None
        self.config = {"workload": f"AllReduce (direct N-way reduction), N=8 fp32, {self.numel} elements "
                                   f"({self.numel * 4 >> 20} MiB) per rank, 8 distinct outputs", "ranks": n,
                       "l2": f"no flush: each step moves {16 * self.numel * 4 >> 30} GiB"}

    def kernels(self):
        b = self.numel * 4
        return [("k_fused_allreduce (no bias, residual or dropout)", "hbm", 2 * self.n * b, 1)]

    def timed(self):
        return self.kernels()

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        if marks:
            marks[0].record(stream)
        coco.coco_allreduce(coco.local(self.inp), coco.replicated(self.out), stream)
        if marks:
            marks[1].record(stream)

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        cnt = rows * 4096
        xs = [synth.as_f64(x[:cnt]) for x in self.inp]
        t0 = time.perf_counter()
        oracle.allreduce(xs)
        return time.perf_counter() - t0, cnt / self.numel


def bert_large_parameter_shapes(layers=24):
    """Parameter shapes of BERT-large (hidden 1024, 24 layers, FFN 4096, 30522-token vocabulary,
    512 positions): about 335 M elements, the size the scattered-tensor section quotes for BERT."""
    h, ffn = 1024, 4096
    shapes = [(30522, h), (512, h), (2, h), (h,), (h,)]
    for _ in range(layers):
        for _ in range(4):  # query, key, value, attention output
            shapes += [(h, h), (h,)]
        shapes += [(h,), (h,), (h, ffn), (ffn,), (ffn, h), (h,), (h,), (h,)]
    shapes += [(h, h), (h,)]  # pooler
    return shapes


class ScatteredGradients(Workload):
    """Data-parallel gradient AllReduce over BERT-large's separately allocated parameter
    tensors, 8 ranks, fp16, in place, averaged (alpha = 1/8)."""

    name = "scattered_allreduce"
    dtype = "f16"

    def __init__(self, dev, n=8, cfg=6, small=False):
        from collective_fusedallreduce_gb300 import coco
        self.n = n
        self.shapes = bert_large_parameter_shapes(6 if small else 24)
        self.grads = [[gen(dev, 100000 * cfg + 1000 * r + t, s, torch.float16, 1e-3) for t, s in enumerate(self.shapes)]
                      for r in range(n)]
        self.numel = sum(int(np.prod(s)) for s in self.shapes)
        nbytes = coco.coco_scattered_table_bytes([int(np.prod(s)) for s in self.shapes], n)
        self.table = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.plan = coco.coco_scattered_table_build(self.grads, self.table)
        self.config = {"workload": f"scattered-tensor AllReduce (CoCoNet): BERT-large parameter list, "
                                   f"{len(self.shapes)} tensors, {self.numel} elements per rank, 8 ranks, fp16, in place, "
                                   f"averaged", "ranks": n, "tensors": len(self.shapes), "elements_per_rank": self.numel,
                       "bucket_table_bytes": nbytes, "l2": "no flush: each step moves 10.7 GB"}

    def kernels(self):
        b = self.numel * 2
        return [("k_scattered_allreduce (1024-element buckets, round-robin over warps)", "hbm",
                 2 * self.n * b + 12 * self.plan.nbuckets * self.n, 1)]

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        if marks:
            marks[0].record(stream)
        coco.coco_scattered_allreduce(self.plan, 1.0 / self.n, stream)
        if marks:
            marks[1].record(stream)

    def rebind(self, key):
        # the bucket table holds the tensors' addresses: one table per buffer set
        from collective_fusedallreduce_gb300 import coco
        if not hasattr(self, "_plans"):
            self._plans = {0: (self.table, self.plan)}
        if key not in self._plans:
            table = torch.empty_like(self.table)
            self._plans[key] = (table, coco.coco_scattered_table_build(self.grads, table))
        self.table, self.plan = self._plans[key]

    def host_inputs(self):
        return [(t, t.cpu().pin_memory()) for row in self.grads for t in row], self.grads[0][0]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        # a sample of whole tensors, in list order, up to `rows` * 4096 elements
        picked, total = [], 0
        for t, s in enumerate(self.shapes):
            if total >= rows * 4096:
                break
            picked.append(t)
            total += int(np.prod(s))
        per_rank = [[synth.as_f64(self.grads[r][t]) for t in picked] for r in range(self.n)]
        t0 = time.perf_counter()
        oracle.scattered_allreduce(per_rank, 1.0 / self.n)
        return time.perf_counter() - t0, total / self.numel

    def full_sample(self):
        return self.numel // 4096


class TinyChain(Workload):
    """The N=2 fp32 configuration: [Decomp] Fig. 2's MLP (x sliced on the batch, W1 column shards, W2 row
    shards: the looped AllGather-Einsum, case 1, then the looped Einsum-ReduceScatter) and a
    FusedAllReduce of two local [4, 16] tensors with bias, dropout p=0.1 and a residual, three calls a
    step. Each call moves a few kilobytes, so the step is launch-bound and its roofline fraction says
    nothing about the kernels; the record carries the step replayed from a CUDA graph beside the eager
    one."""

    name = "tiny_chain"
    dtype = "f32"

    def __init__(self, dev, n=2, b=8, f=16, h=32, p=0.1, seed=0, cfg=1):
        from collective_fusedallreduce_gb300 import synth
        f32 = torch.float32
        self.n, self.b, self.f, self.hd, self.p, self.seed = n, b, f, h, p, seed

        def uni(tid, shape, rank=None):
            sd = synth.seed_of(cfg, tid) if rank is None else synth.seed_of(cfg, tid, rank)
            return synth.tensor(sd, shape, f32, "uniform").to(dev)

        self.x = [uni(0, (b // n, f), r) for r in range(n)]
        self.w1 = [uni(1, (f, h // n), r) for r in range(n)]
        self.w2 = [uni(2, (h // n, f), r) for r in range(n)]
        self.parts = [uni(3, (b // n, f), r) for r in range(n)]
        self.bias = uni(4, (f,))
        self.res = uni(5, (b // n, f))
        self.hbuf = [torch.empty((b, h // n), dtype=f32, device=dev) for _ in range(n)]
        self.y = [torch.empty((b // n, f), dtype=f32, device=dev) for _ in range(n)]
        self.out = [torch.empty((b // n, f), dtype=f32, device=dev) for _ in range(n)]
        self.config = {"workload": "N=2 fp32 chain: Fig. 2 MLP (x[4,16] per rank, W1[16,32] column shards, "
                                   "W2[32,16] row shards; looped AllGather-Einsum case 1, then looped "
                                   "Einsum-ReduceScatter) + FusedAllReduce of 2 local [4,16] + bias[16] + dropout "
                                   "p=0.1 + residual[4,16]; launch-bound (a few KB a call)",
                       "ranks": n, "l2": "not applicable: a few KB a step, launch-bound",
                       "inputs": "synthetic U(-1,1)"}

    def kernels(self):
        n, b, f, hd = self.n, self.b, self.f, self.hd
        e = 4
        ag = ((b * f) + n * (f * hd // n) + n * (b * hd // n)) * e  # gathered x read per rank counted once
        rs = (n * (b * hd // n) + n * (hd // n * f) + n * (b // n * f)) * e
        far = (n * (b // n * f) * 2 + f + b // n * f) * e
        return [("k_gemm_simt (looped AllGather-Einsum, case 1)", "hbm", ag, 1),
                ("k_gemm_simt (looped Einsum-ReduceScatter)", "hbm", rs, 1),
                ("k_fused_allreduce (2 ranks, bias+dropout+residual)", "hbm", far, 1)]

    def step(self, stream, marks=None):
        from collective_fusedallreduce_gb300 import coco
        n = self.n
        if marks:
            marks[0].record(stream)
        coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(self.x, 0), coco.local(self.w1), coco.local(self.hbuf),
                                   stream)
        if marks:
            marks[1].record(stream)
        coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(self.hbuf, 1), coco.sliced(self.w2, 0),
                                   coco.sliced(self.y, 0), stream)
        if marks:
            marks[2].record(stream)
        coco.coco_fused_allreduce(coco.local(self.parts), self.bias, coco.replicated([self.res] * n), self.p,
                                  self.seed, coco.replicated(self.out), stream)
        if marks:
            marks[3].record(stream)

    def graph_seconds(self, stream, steps):
        """The step captured once into a CUDA graph and replayed ``steps`` times (CUDA events)."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=stream.device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            self.step(side)  # warm the plans outside the capture
            with torch.cuda.graph(g, stream=side):
                self.step(side)
        stream.wait_stream(side)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(torch.cuda.current_stream(stream.device))
        for _ in range(steps):
            g.replay()
        e1.record(torch.cuda.current_stream(stream.device))
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1000.0 / steps

    def host_inputs(self):
        ins = [(t, t.cpu().pin_memory()) for t in self.x + self.w1 + self.w2 + self.parts + [self.bias, self.res]]
        return ins, self.out[0]

    def oracle_sample(self, rows):
        import oracle
        from collective_fusedallreduce_gb300 import synth
        x, w1, w2 = ([synth.as_f64(t) for t in ts] for ts in (self.x, self.w1, self.w2))
        parts = [synth.as_f64(t) for t in self.parts]
        b, res = synth.as_f64(self.bias), synth.as_f64(self.res)
        t0 = time.perf_counter()
        oracle.mlp_1d_forward(x, w1, w2)
        oracle.fused_allreduce(parts, b, res, self.p, self.seed)
        return time.perf_counter() - t0, 1.0

    def sample_unit(self):
        return "steps"


WORKLOADS = {"c1": TinyChain, "c2": MegatronTail, "c2o": MegatronTailOverlap, "c2f": MegatronTailFused, "c3": LoopedCase1, "c4a": LoopedCase2, "c4b": LoopedCase3, "c5": Mesh2D,
             "c5b": RsAg, "c5d": AllReduceDirect, "scatter": ScatteredGradients}


# --------------------------------------------------------------- helpers


def host_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def cpu_oracle_rate(wl, peaks, budget_s, min_rows=1):
    """Times the oracle on a sample sized to about ``budget_s``; returns (value, sample text)."""
    rows = max(min_rows, 1)
    dt, frac = wl.oracle_sample(rows)
    while dt < 0.5 and rows < wl.full_sample():
        rows = min(wl.full_sample(), rows * 4)
        dt, frac = wl.oracle_sample(rows)
    if dt < budget_s and rows < wl.full_sample():
        rows = int(min(wl.full_sample(), max(rows, rows * budget_s / max(dt, 1e-3))))
        dt, frac = wl.oracle_sample(rows)
    value = 100.0 * wl.ideal_seconds(peaks) * frac / dt
    return value, dt, rows, frac


def roofline_entry(name, bound, units, avg_s, peaks, traffic, clk=None):
    """The roofline of one timed segment. Tensor-bound kernels are rated against the burst bf16
    figure (a kernel timed by itself, for milliseconds at most); HBM-bound ones against the copy
    figure. When the clock record shows the power cap holding the SM clock down during the timed
    region, the fraction of the sustained bf16 figure (measured in that regime) is added as a note."""
    src = "MEASURED_PEAKS.json" if peaks["source"] == "measured" else "fallback"
    extra = {}
    if bound == "hbm":
        achieved = units / avg_s / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
        src += " (copy)"
    else:
        achieved = units / avg_s / 1e12
        unit = "TFLOP/s"
        peak = peaks["bf16_tflops"]
        src += " (burst)"
        extra["frac_of_burst"] = round(achieved / peak, 4)
        if clk and power_capped_low(clk):
            extra["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
            extra["note"] = (f"sw_power_cap active, median SM clock {clk['sm_mhz']:.0f} of "
                             f"{clk['sm_max_mhz']:.0f} MHz: frac_of_sustained is the fraction of the "
                             f"power-capped bf16 figure")
    return dict({"kernel": name, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                 "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": src}, **extra)


def power_capped_low(clk):
    """The power cap was active and held the median SM clock at least 3 % below its maximum."""
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return "sw_power_cap" in (clk.get("reasons") or []) and bool(sm) and bool(mx) and sm < 0.97 * mx


def load_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) < 4 or line.startswith("#") or parts[0] != kernel_key:
            continue
        src, digest, byts = parts[1], parts[2], parts[3]
        try:
            data = open(os.path.join(ROOT, src), "rb").read()
        except OSError:
            return None
        if hashlib.sha256(data).hexdigest()[:16] != digest:
            return None
        return int(byts)
    return None


# ------------------------------------------------------- multi-GPU helpers


def max_over_ranks(x, dist, device):
    """The largest of every rank's ``x`` (the slowest replica sets the time)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(ideal_s, step_s, world):
    """Whole-job throughput: every replica processes one step's work per ``step_s``."""
    return 100.0 * ideal_s / step_s * world


def measure_e2e(wl, stream, dev, dist, ideal, world, steps):
    """The step end to end through the public calls: every step uploads its inputs from pinned host
    memory and reads its result back, overlapping the compute of other steps; inputs and the result
    are double-buffered, as a data loader would feed the step. A loader packs a step's inputs into one
    pinned staging buffer and the device tensors are views of one device buffer of the same layout, so
    a step's upload is a single copy (one copy per tensor left gaps between the copies: 18 tensors on
    the Megatron tail, 3128 on the BERT-large gradient list). The timed region spans the first upload
    to the last read-back. Two arrangements are timed and the faster reported: uploads and read-backs
    on one copy stream, or on two (concurrent directions)."""
    ins, result = wl.host_inputs()
    devs = [d for d, _ in ins]
    hosts = [h for _, h in ins]
    in_place = any(d is result for d in devs)
    originals = [d.data for d in devs]
    result_original = result.data
    align = 256  # every view starts on a 256-byte boundary, as an allocation would
    sizes = [h.numel() * h.element_size() for h in hosts]
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += -(-n // align) * align
    host_arena = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for h, o, n in zip(hosts, offs, sizes):
        host_arena[o:o + n].copy_(h.reshape(-1).view(torch.uint8))
    del ins, hosts  # the staging buffer holds the inputs now
    arenas = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    sets = [[a[o:o + n].view(d.dtype).view(d.shape) for d, o, n in zip(devs, offs, sizes)] for a in arenas]
    outs = [result.data, None if in_place else torch.empty_like(result)]
    host_out = torch.empty(result.shape, dtype=result.dtype, pin_memory=True)
    h2d = total
    d2h = host_out.numel() * host_out.element_size()
    up = torch.cuda.Stream(device=dev)
    down = up
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]

    def bind(b):
        for d, storage in zip(devs, sets[b]):
            d.data = storage
        if not in_place:
            result.data = outs[b]
        wl.rebind(("e2e", b))

    def upload(b, after_step):
        with torch.cuda.stream(up):
            if after_step:  # set b is free once its last step has computed (and, in place, been read back)
                up.wait_event(downloaded[b] if in_place else computed[b])
            arenas[b].copy_(host_arena, non_blocking=True)
            uploaded[b].record(up)

    def run(n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e0.record(up)
        down.wait_event(e0)
        stream.wait_event(e0)
        upload(0, False)
        if n > 1:
            upload(1, False)
        for k in range(n):
            b = k % 2
            stream.wait_event(uploaded[b])
            if k >= 2:  # the result buffer of step k-2 has been read back
                stream.wait_event(downloaded[b])
            bind(b)
            wl.step(stream)
            computed[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                host_out.copy_(result.data if in_place else outs[b], non_blocking=True)
                downloaded[b].record(down)
            if k + 2 < n:
                upload(b, True)
        e1.record(down)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1000.0

    best = None
    try:
        for mode in ("one copy stream", "two copy streams"):
            down = up if mode == "one copy stream" else torch.cuda.Stream(device=dev)
            run(2)
            et = max_over_ranks(run(steps), dist, dev)
            if best is None or et < best[0]:
                best = (et, mode)
    finally:  # the workload's own tensors again (the staging buffers hold the same values)
        for d, t in zip(devs, originals):
            d.data = t
        result.data = result_original
        wl.rebind(0)
    et, mode = best
    return {"value": aggregate_value(ideal, et / steps, world), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": 1000.0 * et / steps,
            "overlap": f"uploads and read-backs overlap the compute of other steps ({mode}); inputs packed in "
                       "one pinned staging buffer, uploaded by one copy a step; inputs and result double-buffered"}


# ------------------------------------------------------------------- main


def run_reference(args, peaks):
    """The CPU oracle on host cores, K steps of a bounded sample, same metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    wl = WORKLOADS[args.workload](dev)
    # sample size so the whole run stays near ``--reference-seconds``
    dt1, frac1 = wl.oracle_sample(8)
    per_step = max(0.05, args.reference_seconds / max(1, args.steps + args.warmup))
    rows = int(max(1, min(wl.full_sample(), 8 * per_step / max(dt1, 1e-4))))
    for _ in range(args.warmup):
        wl.oracle_sample(rows)
    total, frac = 0.0, 0.0
    for _ in range(args.steps):
        dt, frac = wl.oracle_sample(rows)
        total += dt
    ms = 1000.0 * total / args.steps
    value = 100.0 * wl.ideal_seconds(peaks) * frac / (total / args.steps)
    cores = host_threads()
    sample = f"{rows} of {wl.full_sample()} {wl.sample_unit()} of every rank per step (fraction {frac:.3g} of the workload)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(wl.config),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_steps(wl, stream, dev, dist, steps, warmup, local_rank):
    """Warm-up, then exactly ``steps`` steps timed with CUDA events on the launching stream, bracketed
    by a barrier and a device synchronisation on both sides; clocks sampled meanwhile. Returns the
    slowest rank's step time, the per-segment times (events between a step's calls), the clock
    record and the number of the library's kernel launches in the timed region."""
    from collective_fusedallreduce_gb300 import coco
    kern = wl.timed()
    nk = len(kern)
    for _ in range(warmup):
        wl.step(stream)
    coco.coco_device_status(stream)
    torch.cuda.synchronize()
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = coco.coco_kernel_launches()
    start.record(stream)
    for k in range(steps):
        wl.step(stream, marks[k])
    end.record(stream)
    torch.cuda.synchronize()
    launches = coco.coco_kernel_launches() - launches0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    coco.coco_device_status(stream)  # raises if a bounded device wait gave up
    elapsed = max_over_ranks(start.elapsed_time(end) / 1000.0, dist, dev)
    per_kernel = [sum(marks[k][i].elapsed_time(marks[k][i + 1]) for k in range(steps)) / 1000.0 / steps
                  for i in range(nk)]
    return elapsed / steps, per_kernel, clk, int(launches)


def rooflines(key, wl, per_kernel, peaks, clk):
    """(dominant segment's roofline entry, per-segment breakdown)."""
    kern = wl.timed()
    i_dom = int(np.argmax(per_kernel))
    name, bound, units, _ = kern[i_dom]
    roof = roofline_entry(name, bound, units, per_kernel[i_dom], peaks, load_traffic(f"{key}:{i_dom}"), clk)
    breakdown = []
    for i, (name, bound, units, _) in enumerate(kern):
        e = roofline_entry(name, bound, units, per_kernel[i], peaks, None, clk)
        breakdown.append({"kernel": name, "bound": bound, "us": round(per_kernel[i] * 1e6, 1),
                          "achieved": e["achieved"], "unit": e["unit"], "frac": e["frac"]})
    if hasattr(wl, "flops"):  # an HBM-bound contraction: its tensor-pipe rate beside it
        roof["tensor_tflops"] = round(wl.flops() / per_kernel[i_dom] / 1e12, 1)
        roof["tensor_frac_of_burst"] = round(wl.flops() / per_kernel[i_dom] / 1e12 / peaks["bf16_tflops"], 4)
    return roof, breakdown


# Every configuration besides the headline, each timed in the same process after it (one GPU's
# memory at a time: the previous workload's tensors are freed first).
SUB_CONFIGS = ["c1", "c2", "c3", "c4a", "c4b", "c5", "c5b", "c5d", "scatter"]


def sub_record(key, dev, dist, world, peaks, args, local_rank):
    """One configuration's measurement for the ``configs`` map of the bench line. The step count is
    at least ``--steps`` and enough for about ``--sub-seconds`` of timed work, so that the clock
    record holds samples from under load."""
    wl = WORKLOADS[key](dev)
    stream = torch.cuda.current_stream(dev)
    warm = max(3, args.warmup)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(warm):
        wl.step(stream)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / warm
    est = max_over_ranks(est, dist, dev)
    steps = int(max(args.steps, min(5000, args.sub_seconds / max(est, 1e-6))))
    step_s, per_kernel, clk, launches = time_steps(wl, stream, dev, dist, steps, 3, local_rank)
    roof, breakdown = rooflines(key, wl, per_kernel, peaks, clk)
    ideal = wl.ideal_seconds(peaks)
    rec = {"workload": wl.config["workload"], "dtype": wl.dtype, "steps": steps, "ms_per_step": step_s * 1e3,
           "ideal_ms_per_step": ideal * 1e3, "value": aggregate_value(ideal, step_s, world), "unit": UNIT,
           "kernel": roof["kernel"], "bound": roof["bound"], "achieved": roof["achieved"], "unit_achieved":
           roof["unit"], "frac": roof["frac"], "traffic": roof["traffic"], "roofline": roof, "kernels": breakdown,
           "clocks": clk, "gpu_launches": launches}
    if "frac_of_burst" in roof:
        rec["frac_of_burst"] = roof["frac_of_burst"]
    if hasattr(wl, "graph_seconds"):  # launch-bound: the same step replayed from a CUDA graph
        rec["graph_ms_per_step"] = wl.graph_seconds(stream, steps) * 1e3
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="coco", choices=["coco", "reference"])
    ap.add_argument("--workload", default="c2f", choices=sorted(WORKLOADS))
    ap.add_argument("--configs", default=None,
                    help="comma-separated configurations timed after the headline workload, each a sub-record "
                         "of the line (default: every other configuration when the headline is the default "
                         "workload; 'none' for none)")
    ap.add_argument("--sub-seconds", type=float, default=0.25,
                    help="timed work per sub-record, at least --steps steps")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    ap.add_argument("--small", action="store_true",
                    help="reduced size of the c5b and scatter workloads (a few GB on the device, for ncu)")
    args = ap.parse_args()
    peaks = load_peaks()

    if args.impl == "reference":
        return run_reference(args, peaks)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()

    if args.configs is None:
        subs = [c for c in SUB_CONFIGS if c != args.workload] if args.workload == "c2f" else []
    elif args.configs == "none":
        subs = []
    else:
        subs = [c for c in args.configs.split(",") if c]
        for c in subs:
            if c not in WORKLOADS:
                raise SystemExit(f"unknown configuration {c!r}")

    wl = WORKLOADS[args.workload](dev, **({"small": True} if args.small and args.workload in ("c5b", "c5d", "scatter") else {}))
    stream = torch.cuda.current_stream(dev)
    step_s, per_kernel, clk, launches = time_steps(wl, stream, dev, dist, args.steps, args.warmup, local_rank)
    ideal = wl.ideal_seconds(peaks)
    value = aggregate_value(ideal, step_s, world)
    roof, breakdown = rooflines(args.workload, wl, per_kernel, peaks, clk)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1000.0, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded torch CUDA generator)",
            "config": dict(wl.config, parallelism=f"{wl.config.get('ranks', 8)} logical ranks in one GPU"
                           + (f" x {world} replicas" if world > 1 else "")),
            "roofline": roof, "kernels": breakdown, "gpu_launches": launches, "clocks": clk,
            "ideal_ms_per_step": ideal * 1000.0}

    # end to end: host buffers in, result back, through the same public calls
    if not args.no_e2e:
        line["e2e"] = measure_e2e(wl, stream, dev, dist, ideal, world, max(3, min(args.steps, 50)))

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, rows, frac = cpu_oracle_rate(wl, peaks, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": host_threads(), "kind": "oracle",
                                "sample": f"{rows} of {wl.full_sample()} {wl.sample_unit()} of every rank, one pass, "
                                          f"{dt:.2f} s (fraction {frac:.3g} of one step)"}
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if subs:
        line["configs"] = {c: sub_record(c, dev, dist, world, peaks, args, local_rank) for c in subs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
