"""coco_einsum_accumulate: out += lhs @ rhs with the Addition in the einsum's epilogue, against the
float64 oracle (the einsum plus the output's former values), through the C-ABI."""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import coco, synth
from helpers import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _dev(ts):
    return [t.to(DEV) for t in ts]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("n,m,k,nn", [(1, 128, 64, 256), (4, 264, 128, 320), (8, 200, 512, 136), (2, 384, 1000, 264)])
def test_matches_the_oracle(dtype, n, m, k, nn):
    lhs = synth.per_rank(501, 0, n, (m, k), dtype, std=k ** -0.5)
    rhs = synth.per_rank(501, 1, n, (k, nn), dtype)
    out0 = synth.per_rank(501, 2, n, (m, nn), torch.float32)
    out = _dev(out0)
    coco.coco_einsum_accumulate("mk,kn->mn", coco.local(_dev(lhs)), coco.local(_dev(rhs)), coco.local(out))
    coco.coco_device_status()
    for r in range(n):
        want = synth.as_f64(out0[r]) + oracle.einsum("mk,kn->mn", synth.as_f64(lhs[r]), synth.as_f64(rhs[r]))
        assert_close(out[r], want, dtype, f"rank {r}")


@pytest.mark.parametrize("k", [64, 512])
def test_small_integers_are_exact_and_repeat(k):
    """Every sum exact: the result equals the float64 one bit for bit; a second call (the cached plan)
    adds the product again."""
    n, m, nn = 4, 256, 256
    lhs = synth.per_rank(502, 0, n, (m, k), torch.bfloat16, "smallint")
    rhs = synth.per_rank(502, 1, n, (k, nn), torch.bfloat16, "smallint")
    out0 = synth.per_rank(502, 2, n, (m, nn), torch.float32, "smallint")
    out = _dev(out0)
    dl, dr = _dev(lhs), _dev(rhs)
    for times in (1, 2):
        coco.coco_einsum_accumulate("mk,kn->mn", coco.local(dl), coco.local(dr), coco.local(out))
        coco.coco_device_status()
        for r in range(n):
            prod = oracle.einsum("mk,kn->mn", synth.as_f64(lhs[r]), synth.as_f64(rhs[r]))
            assert np.array_equal(synth.as_f64(out[r]), synth.as_f64(out0[r]) + times * prod)


def test_batched_and_fp32_operands():
    n, b, m, k, nn = 2, 3, 128, 96, 136
    lhs = synth.per_rank(503, 0, n, (b, m, k), torch.bfloat16)
    rhs = synth.per_rank(503, 1, n, (b, k, nn), torch.bfloat16)
    out0 = synth.per_rank(503, 2, n, (b, m, nn), torch.float32)
    out = _dev(out0)
    coco.coco_einsum_accumulate("bmk,bkn->bmn", coco.local(_dev(lhs)), coco.local(_dev(rhs)), coco.local(out))
    coco.coco_device_status()
    for r in range(n):
        want = synth.as_f64(out0[r]) + oracle.einsum("bmk,bkn->bmn", synth.as_f64(lhs[r]), synth.as_f64(rhs[r]))
        assert_close(out[r], want, torch.bfloat16, f"batched rank {r}")
    # fp32 operands: the FMA path, at the fp32 tolerance
    lhs = synth.per_rank(503, 3, n, (40, 24), torch.float32, "uniform")
    rhs = synth.per_rank(503, 4, n, (24, 16), torch.float32, "uniform")
    out0 = synth.per_rank(503, 5, n, (40, 16), torch.float32, "uniform")
    out = _dev(out0)
    coco.coco_einsum_accumulate("mk,kn->mn", coco.local(_dev(lhs)), coco.local(_dev(rhs)), coco.local(out))
    coco.coco_device_status()
    for r in range(n):
        want = synth.as_f64(out0[r]) + oracle.einsum("mk,kn->mn", synth.as_f64(lhs[r]), synth.as_f64(rhs[r]))
        assert_close(out[r], want, torch.float32, f"fp32 rank {r}")


def test_empty_contraction_leaves_the_output():
    out0 = torch.randn(2, 64, 64)
    out = [o.to(DEV) for o in out0]
    lhs = [torch.empty((64, 0), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    rhs = [torch.empty((0, 64), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    coco.coco_einsum_accumulate("mk,kn->mn", coco.local(lhs), coco.local(rhs), coco.local(out))
    torch.cuda.synchronize()
    for a, b in zip(out, out0):
        assert torch.equal(a.cpu(), b)
