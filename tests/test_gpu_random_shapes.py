"""Seeded random sweep over the looped einsums: shapes, rank counts and dtypes drawn at random (multiples
of 8 elements, so every call is valid), spanning both tensor-core variants (short K: one CTA per MMA;
longer K: the CTA-pair MMA) and ragged tile tails, each compared with the oracle within the tolerance of
its output dtype. The fixed seeds make every case reproducible."""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, dev, empty_like_list, f64

pytestmark = pytest.mark.gpu

BF16, F16, F32 = torch.bfloat16, torch.float16, torch.float32
KINDS = ["case1", "case2", "case3", "rs_m", "rs_n"]


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


def draw(seed):
    rng = np.random.default_rng(10_000 + seed)
    kind = KINDS[seed % len(KINDS)]
    n = int(rng.choice([1, 2, 3, 4, 5, 8]))
    dtype = [BF16, F16][int(rng.integers(2))]
    mul8 = lambda lo, hi: 8 * int(rng.integers(lo // 8, hi // 8 + 1))
    return rng, kind, n, dtype, mul8


@pytest.mark.parametrize("seed", range(50))
def test_random_looped_einsum(coco, seed):
    rng, kind, n, dtype, mul8 = draw(seed)
    cfg = 60 + seed
    if kind == "case1":
        ms, k, nn = mul8(8, 320), mul8(64, 1024), mul8(8, 640)
        shards = synth.per_rank(cfg, 0, n, (ms, k), dtype, std=k ** -0.5)
        rhs = synth.per_rank(cfg, 1, n, (k, nn), dtype)
        outs = empty_like_list(n, (n * ms, nn), dtype)
        coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 0), coco.local(dev(rhs)), coco.local(outs))
        refs = oracle.allgather_einsum("mk,kn->mn", "lhs", "m", [f64(s) for s in shards], [f64(x) for x in rhs])
        out_dtype = dtype
    elif kind == "case2":
        m, ks, nn = mul8(8, 640), mul8(8, 256), mul8(8, 640)
        out_dtype = [F32, dtype][int(rng.integers(2))]
        shards = synth.per_rank(cfg, 0, n, (m, ks), dtype, std=(n * ks) ** -0.5)
        rhs = synth.per_rank(cfg, 1, n, (n * ks, nn), dtype)
        outs = empty_like_list(n, (m, nn), out_dtype)
        coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(dev(shards), 1), coco.local(dev(rhs)), coco.local(outs))
        refs = oracle.allgather_einsum("mk,kn->mn", "lhs", "k", [f64(s) for s in shards], [f64(x) for x in rhs])
    elif kind == "case3":
        bs, m, k, nn = int(rng.integers(1, 4)), mul8(8, 400), mul8(64, 512), mul8(8, 400)
        shards = synth.per_rank(cfg, 0, n, (bs, m, k), dtype, std=k ** -0.5)
        rhs = synth.per_rank(cfg, 1, n, (n * bs, k, nn), dtype)
        outs = empty_like_list(n, (n * bs, m, nn), dtype)
        coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.sliced(dev(shards), 0), coco.local(dev(rhs)),
                                   coco.local(outs))
        refs = oracle.allgather_einsum("bmk,bkn->bmn", "lhs", "b", [f64(s) for s in shards], [f64(x) for x in rhs])
        out_dtype = dtype
    else:
        label = kind[-1]
        ks = mul8(8, 256)
        m = n * mul8(8, 160) if label == "m" else mul8(8, 480)
        nn = n * mul8(8, 160) if label == "n" else mul8(8, 480)
        lhs = synth.per_rank(cfg, 0, n, (m, ks), dtype, std=(n * ks) ** -0.5)
        rhs = synth.per_rank(cfg, 1, n, (ks, nn), dtype)
        shape = (m // n, nn) if label == "m" else (m, nn // n)
        outs = empty_like_list(n, shape, dtype)
        coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(dev(lhs), 1), coco.sliced(dev(rhs), 0),
                                   coco.sliced(outs, 0 if label == "m" else 1))
        refs = oracle.einsum_reduce_scatter("mk,kn->mn", [f64(x) for x in lhs], [f64(x) for x in rhs], label)
        out_dtype = dtype
    coco.coco_device_status()
    torch.cuda.synchronize()
    for r, (o, ref) in enumerate(zip(outs, refs)):
        assert_close(o, ref, out_dtype, f"seed {seed} {kind} n={n} {dtype} rank {r}")


@pytest.mark.parametrize("seed", range(30))
def test_random_fused_allreduce(coco, seed):
    """Random shape, rank count, dtype, dropout probability, with or without bias and residual, distinct
    or aliased outputs."""
    rng = np.random.default_rng(20_000 + seed)
    n = int(rng.choice([1, 2, 3, 4, 8]))
    dtype = [F32, F16, BF16][seed % 3]
    ndim = int(rng.integers(1, 4))
    shape = tuple(int(x) for x in rng.integers(1, 40, ndim - 1)) + (8 * int(rng.integers(1, 200)),)
    p = float(rng.choice([0.0, 0.1, 0.5]))
    seed_hash = int(rng.integers(0, 2 ** 63))
    cfg = 120 + seed
    parts = synth.per_rank(cfg, 0, n, shape, dtype, "uniform")
    bias = synth.tensor(synth.seed_of(cfg, 1), (shape[-1],), dtype, "uniform") if rng.integers(2) else None
    res = synth.tensor(synth.seed_of(cfg, 2), shape, dtype, "uniform") if rng.integers(2) else None
    aliased = bool(rng.integers(2))
    outs = empty_like_list(1 if aliased else n, shape, dtype)
    out_list = outs * n if aliased else outs
    coco.coco_fused_allreduce(coco.local(dev(parts)), None if bias is None else bias.cuda(),
                              None if res is None else coco.replicated([res.cuda()] * n), p, seed_hash,
                              coco.replicated(out_list))
    ref = oracle.fused_allreduce([f64(x) for x in parts], None if bias is None else f64(bias),
                                 None if res is None else f64(res), p, seed_hash)
    coco.coco_device_status()
    for r, o in enumerate(outs):
        assert_close(o, ref, dtype, f"seed {seed} n={n} {dtype} {shape} p={p} rank {r}")


@pytest.mark.parametrize("seed", range(20))
def test_random_matmul_fused_allreduce(coco, seed):
    rng = np.random.default_rng(30_000 + seed)
    n = int(rng.choice([1, 2, 4, 8]))
    dtype = [F16, BF16][seed % 2]
    rows = 8 * int(rng.integers(1, 80))
    ks = 8 * int(rng.integers(2, 40))
    hid = 8 * int(rng.integers(1, 100))
    p = float(rng.choice([0.0, 0.1]))
    cfg = 160 + seed
    ins = synth.per_rank(cfg, 0, n, (rows, ks), dtype)
    ws = synth.per_rank(cfg, 1, n, (ks, hid), dtype, std=(n * ks) ** -0.5)
    bias = synth.tensor(synth.seed_of(cfg, 2), (hid,), dtype, std=0.02)
    res = synth.tensor(synth.seed_of(cfg, 3), (rows, hid), dtype)
    outs = empty_like_list(n, (rows, hid), dtype)
    coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(dev(ins), 1), coco.sliced(dev(ws), 0), bias.cuda(),
                                     coco.replicated([res.cuda()] * n), p, 99 + seed, coco.replicated(outs))
    ref = oracle.megatron_attention_tail([f64(x) for x in ins], [f64(w) for w in ws], f64(bias), f64(res), p,
                                         99 + seed)[1]
    coco.coco_device_status()
    for r, o in enumerate(outs):
        assert_close(o, ref, dtype, f"seed {seed} n={n} {dtype} rows={rows} ks={ks} hid={hid} rank {r}")
