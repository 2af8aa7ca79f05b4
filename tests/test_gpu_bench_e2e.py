"""The end-to-end measurement of bench.py feeds the same public calls from one packed pinned staging
buffer per step. Afterwards the workload's tensors are its own again, and a step gives the same bits
as before it; the reported upload size is the packed inputs (each view 256-byte aligned)."""

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bench():
    import __graft_entry__
    __graft_entry__.build()
    import bench as b
    return b


def _device_inputs(name, wl):
    if name == "c1":
        return wl.x + wl.w1 + wl.w2 + wl.parts + [wl.bias, wl.res], wl.out[0]
    if name == "c2":
        return wl.inp + wl.w + [wl.bias, wl.res], wl.out[0]
    if name == "c4b":
        return wl.l + wl.r, wl.out[0]
    return [t for row in wl.grads for t in row], wl.grads[0][0]  # scatter: in place


@pytest.mark.parametrize("name", ["c1", "c2", "c4b", "scatter"])
def test_e2e_restores_the_workload_and_keeps_its_results(bench, name):
    dev = torch.device("cuda", 0)
    wl = bench.WORKLOADS[name](dev)
    stream = torch.cuda.current_stream(dev)
    wl.step(stream)  # the averaged gradients are a fixed point of the in-place AllReduce
    devs, result = _device_inputs(name, wl)
    ptrs = [d.data_ptr() for d in devs]
    result_ptr = result.data_ptr()
    nbytes = sum(d.numel() * d.element_size() for d in devs)
    torch.cuda.synchronize()
    ref = result.clone()

    e = bench.measure_e2e(wl, stream, dev, None, 1e-3, 1, 3)

    assert [d.data_ptr() for d in devs] == ptrs
    assert result.data_ptr() == result_ptr
    assert nbytes <= e["h2d_bytes_per_step"] < nbytes + 256 * len(devs)
    assert e["d2h_bytes_per_step"] == result.numel() * result.element_size()
    assert e["ms_per_step"] > 0
    wl.step(stream)
    torch.cuda.synchronize()
    assert torch.equal(result, ref)


def test_tiny_chain_graph_replay_gives_the_eager_bits(bench):
    # the N=2 fp32 configuration is launch-bound; its record adds the step replayed from a CUDA graph
    dev = torch.device("cuda", 0)
    wl = bench.WORKLOADS["c1"](dev)
    stream = torch.cuda.current_stream(dev)
    wl.step(stream)
    torch.cuda.synchronize()
    eager = [t.clone() for t in wl.y + wl.out]
    for t in wl.y + wl.out:
        t.fill_(float("nan"))
    assert wl.graph_seconds(stream, 5) > 0
    for a, b in zip(wl.y + wl.out, eager):
        assert torch.equal(a, b)
