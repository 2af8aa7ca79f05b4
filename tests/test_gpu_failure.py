"""The device-side failure path on a GB300, without a fault: a bounded wait on an mbarrier phase
that nothing completes gives up after its limit, the kernel records COCO_ERR_TIMEOUT, frees its
tensor memory and returns; the host reads the status once and the context stays usable."""

import time

import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, dev, empty_like_list, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


def test_bounded_wait_reports_timeout_and_the_context_stays_usable(coco):
    coco.coco_device_status()  # nothing pending
    t0 = time.perf_counter()
    coco.coco_wait_selftest(2_000_000)  # 2 ms limit
    with pytest.raises(coco.CocoError) as exc:
        coco.coco_device_status()
    assert exc.value.name == "COCO_ERR_TIMEOUT"
    assert time.perf_counter() - t0 < 10.0
    coco.coco_device_status()  # reported once, then cleared
    # the context still runs work: a small FusedAllReduce against the oracle
    n, shape = 4, (16, 64)
    parts = synth.per_rank(35, 0, n, shape, torch.float16, "uniform")
    outs = empty_like_list(n, shape, torch.float16)
    coco.coco_fused_allreduce(coco.local(dev(parts)), None, None, 0.1, 3, coco.replicated(outs))
    coco.coco_device_status()
    ref = oracle.fused_allreduce([f64(x) for x in parts], None, None, 0.1, 3)
    for o in outs:
        assert_close(o, ref, torch.float16)


def test_timeouts_repeat_and_stay_bounded(coco):
    for limit in (1_000, 100_000, 10_000_000):
        t0 = time.perf_counter()
        coco.coco_wait_selftest(limit)
        with pytest.raises(coco.CocoError) as exc:
            coco.coco_device_status()
        assert exc.value.name == "COCO_ERR_TIMEOUT"
        assert time.perf_counter() - t0 < 10.0
    coco.coco_device_status()
