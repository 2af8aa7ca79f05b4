"""Every entry point is stream-ordered and never synchronises with the host, so a sequence of calls
can be captured into a CUDA graph once and replayed: the replays give the same bits as eager calls.

Covered: the FusedAllReduce (dropout on), the RS-AG split, looped AllGather-Einsum case 1, case 2 with a
long K loop (the launch whose producers wait for each other between waves, a cooperative launch), the
looped Einsum-ReduceScatter, the fused MatMul + FusedAllReduce, the in-place scattered-tensor AllReduce
and the 2-D mesh MLP with its AllGather on a second stream.
"""

import pytest
import torch

from collective_fusedallreduce_gb300 import synth

pytestmark = pytest.mark.gpu

BF16, F16, F32 = torch.bfloat16, torch.float16, torch.float32


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


def per_rank(cfg, tid, n, shape, dtype, std=1.0):
    return [t.cuda() for t in synth.per_rank(cfg, tid, n, shape, dtype, std=std)]


def eager_then_graph(coco, run, outs, inputs=()):
    """Runs `run` eagerly, snapshots `outs`, captures `run` into a graph and replays it twice on fresh
    output buffers (and, for in-place calls, on the original `inputs` restored first). Returns the
    eager and replayed snapshots."""
    saved = [t.clone() for t in inputs]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up off the capture: first-call attributes and plans
        run()
    torch.cuda.current_stream().wait_stream(side)
    coco.coco_device_status()
    for t, s in zip(inputs, saved):
        t.copy_(s)
    torch.cuda.synchronize()
    run()
    coco.coco_device_status()
    eager = [t.clone() for t in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    replays = []
    for _ in range(2):
        for t in outs:
            t.fill_(float("nan")) if t.is_floating_point() else t.zero_()
        for t, s in zip(inputs, saved):
            t.copy_(s)
        g.replay()
        torch.cuda.synchronize()
        coco.coco_device_status()
        replays.append([t.clone() for t in outs])
    return eager, replays


def assert_same(eager, replays):
    for rep in replays:
        for i, (a, b) in enumerate(zip(eager, rep)):
            assert torch.equal(a, b), f"output {i} differs after replay"


def test_fused_allreduce_graph(coco):
    n, rows, cols = 8, 1024, 1536
    parts = per_rank(40, 0, n, (rows, cols), F16)
    bias = per_rank(40, 1, 1, (cols,), F16, std=0.02)[0]
    res = per_rank(40, 2, 1, (rows, cols), F16)[0]
    outs = [torch.empty(rows, cols, dtype=F16, device="cuda") for _ in range(n)]
    run = lambda: coco.coco_fused_allreduce(coco.local(parts), bias, coco.replicated([res] * n), 0.1, 77,
                                            coco.replicated(outs))
    assert_same(*eager_then_graph(coco, run, outs))


def test_rs_ag_graph(coco):
    n, numel = 8, 1 << 20
    inp = per_rank(41, 0, n, (numel,), F32)
    scratch = [torch.empty(numel // n, device="cuda") for _ in range(n)]
    outs = [torch.empty(numel, device="cuda") for _ in range(n)]
    run = lambda: coco.coco_allreduce_rs_ag(coco.local(inp), coco.sliced(scratch, 0), coco.replicated(outs))
    assert_same(*eager_then_graph(coco, run, outs))


def test_looped_ag_einsum_case1_graph(coco):
    n, m, k, nn = 4, 1024, 1024, 768
    shards = per_rank(42, 0, n, (m // n, k), BF16, std=k ** -0.5)
    b = per_rank(42, 1, n, (k, nn), BF16)
    outs = [torch.empty(m, nn, dtype=BF16, device="cuda") for _ in range(n)]
    run = lambda: coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(shards, 0), coco.local(b), coco.local(outs))
    assert_same(*eager_then_graph(coco, run, outs))


def test_looped_ag_einsum_case2_long_k_graph(coco):
    """K = 8192 and a 128 MiB B operand per rank: the producers of this launch wait for each other
    between waves, so it is launched cooperatively; the capture keeps that launch and the reset of its
    arrival counter."""
    n, m, k, nn = 2, 1024, 8192, 8192
    a = per_rank(43, 0, n, (m, k // n), BF16, std=k ** -0.5)
    rhs = per_rank(43, 1, n, (k, nn), BF16)
    outs = [torch.empty(m, nn, dtype=F32, device="cuda") for _ in range(n)]
    run = lambda: coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(a, 1), coco.local(rhs), coco.local(outs))
    assert_same(*eager_then_graph(coco, run, outs))


def test_looped_einsum_rs_graph(coco):
    n, m, k, nn = 4, 512, 2048, 1024
    lhs = per_rank(44, 0, n, (m, k // n), BF16, std=k ** -0.5)
    rhs = per_rank(44, 1, n, (k // n, nn), BF16)
    outs = [torch.empty(m // n, nn, dtype=BF16, device="cuda") for _ in range(n)]
    run = lambda: coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(lhs, 1), coco.sliced(rhs, 0),
                                             coco.sliced(outs, 0))
    assert_same(*eager_then_graph(coco, run, outs))


def test_matmul_fused_allreduce_graph(coco):
    n, rows, hidden = 8, 512, 1024
    ins = per_rank(45, 0, n, (rows, hidden // n), F16)
    ws = per_rank(45, 1, n, (hidden // n, hidden), F16, std=0.02)
    bias = per_rank(45, 2, 1, (hidden,), F16, std=0.02)[0]
    res = per_rank(45, 3, 1, (rows, hidden), F16)[0]
    outs = [torch.empty(rows, hidden, dtype=F16, device="cuda") for _ in range(n)]
    run = lambda: coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(ins, 1), coco.sliced(ws, 0), bias,
                                                   coco.replicated([res] * n), 0.1, 5, coco.replicated(outs))
    assert_same(*eager_then_graph(coco, run, outs))


def test_scattered_allreduce_graph(coco):
    """In place: every replay starts from the same gradients, restored by copies inside the replay loop."""
    n = 4
    shapes = [(300, 7), (1024,), (5, 5, 40), (1,), (2048, 3)]
    grads = [[t.cuda() for t in synth.per_rank(46, i, n, s, F16)] for i, s in enumerate(shapes)]
    grads = [[grads[t][r] for t in range(len(shapes))] for r in range(n)]
    nbytes = coco.coco_scattered_table_bytes([int(torch.tensor(s).prod()) for s in shapes], n)
    table = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    plan = coco.coco_scattered_table_build(grads, table)
    flat = [t for row in grads for t in row]
    run = lambda: coco.coco_scattered_allreduce(plan, 1.0 / n)
    assert_same(*eager_then_graph(coco, run, flat, inputs=flat))


def test_mesh_2d_mlp_graph(coco):
    """Two streams inside the capture: the AllGather of W2 forks onto a side stream and joins back."""
    from collective_fusedallreduce_gb300 import workloads
    m_x, n_y = 2, 4
    b, f, h = 64 * n_y, 64 * m_x * n_y, 128 * m_x
    keys = [(x, y) for x in range(m_x) for y in range(n_y)]
    xb = {k: synth.tensor(synth.seed_of(47, 0, i), (b // n_y, f // m_x), BF16).cuda() for i, k in enumerate(keys)}
    w1 = {k: synth.tensor(synth.seed_of(47, 1, i), (f // n_y, h // m_x), BF16, std=f ** -0.5).cuda()
          for i, k in enumerate(keys)}
    w2 = {k: synth.tensor(synth.seed_of(47, 2, i), (h // m_x, f // n_y), BF16, std=h ** -0.5).cuda()
          for i, k in enumerate(keys)}
    bufs = workloads.mlp_2d(xb, w1, w2, m_x, n_y)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    outs = [bufs[name][k] for name in ("xf", "h", "w2f", "y") for k in keys]
    run = lambda: workloads.mlp_2d(xb, w1, w2, m_x, n_y, bufs, side_stream=side)
    assert_same(*eager_then_graph(coco, run, outs))


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_scattered_table_build_is_refused_under_capture(coco):
    """The table upload reads a host buffer freed when the call returns, which a graph would replay."""
    n = 2
    grads = [[t.cuda() for t in synth.per_rank(48, 0, n, (4096,), F16)]]
    grads = [[grads[0][r]] for r in range(n)]
    table = torch.empty(coco.coco_scattered_table_bytes([4096], n), dtype=torch.uint8, device="cuda")
    g = torch.cuda.CUDAGraph()
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        with torch.cuda.graph(g):
            coco.coco_scattered_table_build(grads, table)
    plan = coco.coco_scattered_table_build(grads, table)  # outside capture it works
    coco.coco_scattered_allreduce(plan, 0.5)
    torch.cuda.synchronize()
    coco.coco_device_status()
