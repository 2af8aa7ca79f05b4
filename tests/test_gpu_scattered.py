"""GPU parity of the scattered-tensor AllReduce ([CoCoNet], scattered tensors).

Lists of separately allocated tensors of mixed sizes (empty, single element,
ragged against the 1024-element buckets, large) are reduced in place on every
rank and compared with the oracle's plain per-tensor definition.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


SIZES = [(7,), (1,), (0,), (1023,), (1024,), (1025,), (3, 5000), (64, 1000), (100003,)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 2, 3, 8])
@pytest.mark.parametrize("alpha", [1.0, 0.125])
def test_scattered_allreduce_matches_oracle(coco, dtype, n, alpha):
    host = [[synth.tensor(synth.seed_of(40, t, r), s, dtype, "uniform") for t, s in enumerate(SIZES)] for r in range(n)]
    dev = [[x.cuda() for x in row] for row in host]
    nbytes = coco.coco_scattered_table_bytes([x.numel() for x in host[0]], n)
    table = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    plan = coco.coco_scattered_table_build(dev, table)
    assert plan.nbuckets == sum(-(-x.numel() // 1024) for x in host[0])
    coco.coco_scattered_allreduce(plan, alpha)
    torch.cuda.synchronize()
    ref = oracle.scattered_allreduce([[f64(x) for x in row] for row in host], alpha)
    for r in range(n):
        for t in range(len(SIZES)):
            assert_close(dev[r][t], ref[t], dtype, f"rank {r} tensor {t}")
            assert torch.equal(dev[r][t], dev[0][t])  # every rank holds the same values


def test_table_is_reusable_across_steps(coco):
    n = 4
    dev = [[torch.full(s, float(r + 1), device="cuda") for s in SIZES] for r in range(n)]
    table = torch.empty(coco.coco_scattered_table_bytes([x.numel() for x in dev[0]], n), dtype=torch.uint8,
                        device="cuda")
    plan = coco.coco_scattered_table_build(dev, table)
    for step in range(3):  # in place, averaged: the values stay at the mean 2.5
        coco.coco_scattered_allreduce(plan, 1.0 / n)
    torch.cuda.synchronize()
    for row in dev:
        for x in row:
            assert torch.all(x == 2.5)


def test_table_metadata_size_follows_the_page(coco):
    # 12 bytes per bucket of at most 1024 elements, per rank
    for numels, n in [([334000000], 1), ([1, 1024, 1025], 8)]:
        got = coco.coco_scattered_table_bytes(numels, n)
        assert got - 64 == n * sum(oracle.scattered_metadata_bytes(x) for x in numels)
