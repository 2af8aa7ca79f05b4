"""GPU parity of the composite workloads and of every configuration at full size.

Small forms run the whole chain and compare every output with the oracle; the
``slow`` tests run the full-size configurations in the launch configuration
``bench.py`` times (same shapes, one call per step) and compare sampled rows,
which the oracle computes from the same input values copied to the host.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, dev, f64

pytestmark = pytest.mark.gpu

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


def test_config1_mlp_fig2_chain(coco, workloads):
    """N=2 fp32 U(-1,1): x[B/N=4, F=16] per rank, W1[16,32] column shards, W2[32,16] row shards;
    looped AllGather-Einsum (case 1) then looped Einsum-ReduceScatter."""
    n, b, f, h = 2, 8, 16, 32
    x = synth.per_rank(1, 0, n, (b // n, f), F32, "uniform")
    w1 = synth.per_rank(1, 1, n, (f, h // n), F32, "uniform")
    w2 = synth.per_rank(1, 2, n, (h // n, f), F32, "uniform")
    hs, ys = workloads.mlp_1d(dev(x), dev(w1), dev(w2))
    coco.coco_device_status()
    ref_y = oracle.mlp_1d_forward([f64(a) for a in x], [f64(a) for a in w1], [f64(a) for a in w2])
    ref_h = oracle.looped_allgather_einsum("mk,kn->mn", "lhs", "m", [f64(a) for a in x], [f64(a) for a in w1])
    for r in range(n):
        assert_close(hs[r], ref_h[r], F32, f"h rank {r}")
        assert_close(ys[r], ref_y[r], F32, f"y rank {r}")
    # and the whole chain equals the unpartitioned MLP on the gathered batch
    full = oracle.mlp_1d_reference(np.concatenate([f64(a) for a in x]), np.concatenate([f64(a) for a in w1], 1),
                                   np.concatenate([f64(a) for a in w2], 0))
    assert_close(torch.cat([y.cpu() for y in ys]), full, F32, "y vs unpartitioned")


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_megatron_tail_chain_small(coco, workloads, dtype):
    n, rows, hidden = 8, 264, 512
    ins = synth.per_rank(2, 10, n, (rows, hidden // n), dtype)
    ws = synth.per_rank(2, 11, n, (hidden // n, hidden), dtype, std=0.02)
    bias = synth.tensor(synth.seed_of(2, 12), (hidden,), dtype, std=0.02)
    res = synth.tensor(synth.seed_of(2, 13), (rows, hidden), dtype)
    _, out = workloads.megatron_attention_tail(dev(ins), dev(ws), bias.cuda(), res.cuda(), 0.1, 5)
    torch.cuda.synchronize()
    _, ref = oracle.megatron_attention_tail([f64(a) for a in ins], [f64(w) for w in ws], f64(bias), f64(res), 0.1, 5)
    for q, o in enumerate(out):
        assert_close(o, ref, dtype, f"rank {q}")


@pytest.mark.parametrize("chunks", [1, 3, 4, 7])
def test_megatron_tail_overlap_equals_the_unchunked_chain(coco, workloads, chunks):
    """[CoCoNet] §5.3 Overlap in row chunks on two streams: bit for bit the unchunked chain's
    partials and outputs (the chunks' FusedAllReduces continue the dropout index)."""
    n, rows, hidden = 8, 264, 512
    ins = dev(synth.per_rank(2, 20, n, (rows, hidden // n), F16))
    ws = dev(synth.per_rank(2, 21, n, (hidden // n, hidden), F16, std=0.02))
    bias = synth.tensor(synth.seed_of(2, 22), (hidden,), F16, std=0.02).cuda()
    res = synth.tensor(synth.seed_of(2, 23), (rows, hidden), F16).cuda()
    layer_a, out_a = workloads.megatron_attention_tail(ins, ws, bias, res, 0.1, 9)
    side = torch.cuda.Stream()
    layer_b = out_b = None
    for _ in range(2):  # twice: the second call reuses the buffers the first one's side stream wrote
        layer_b, out_b = workloads.megatron_attention_tail_overlap(ins, ws, bias, res, 0.1, 9, chunks, layer_b, out_b,
                                                                   side_stream=side)
    coco.coco_device_status()
    for q in range(n):
        assert torch.equal(layer_a[q], layer_b[q])
        assert torch.equal(out_a[q], out_b[q])


def test_mesh_2d_mlp_side_stream_gives_the_same_bits(coco, workloads):
    """The AllGather of W2 on a second stream beside the first einsum: the same outputs, bit for bit,
    twice in a row (the second call's AllGather waits for the first call's reads of its buffer)."""
    m_x, n_y = 2, 4
    b, f, h = 64 * n_y, 64 * m_x * n_y, 128 * m_x
    keys = [(x, y) for x in range(m_x) for y in range(n_y)]
    xb = {k: synth.tensor(synth.seed_of(5, 3, i), (b // n_y, f // m_x), BF16).cuda() for i, k in enumerate(keys)}
    w1 = {k: synth.tensor(synth.seed_of(5, 4, i), (f // n_y, h // m_x), BF16, std=f ** -0.5).cuda()
          for i, k in enumerate(keys)}
    w2 = {k: synth.tensor(synth.seed_of(5, 5, i), (h // m_x, f // n_y), BF16, std=h ** -0.5).cuda()
          for i, k in enumerate(keys)}
    one = workloads.mlp_2d(xb, w1, w2, m_x, n_y)
    side = torch.cuda.Stream()
    two = None
    for _ in range(2):
        two = workloads.mlp_2d(xb, w1, w2, m_x, n_y, two, side_stream=side)
    coco.coco_device_status()
    for name in ("xf", "h", "w2f", "y"):
        for k in keys:
            assert torch.equal(one[name][k], two[name][k]), (name, k)


@pytest.mark.parametrize("m_x,n_y", [(2, 4), (1, 2), (2, 1)])
def test_mesh_2d_mlp_small(coco, workloads, m_x, n_y):
    b, f, h = 64 * n_y, 64 * m_x * n_y, 128 * m_x
    keys = [(x, y) for x in range(m_x) for y in range(n_y)]
    xb = {k: synth.tensor(synth.seed_of(5, 0, i), (b // n_y, f // m_x), BF16) for i, k in enumerate(keys)}
    w1 = {k: synth.tensor(synth.seed_of(5, 1, i), (f // n_y, h // m_x), BF16, std=f ** -0.5) for i, k in enumerate(keys)}
    w2 = {k: synth.tensor(synth.seed_of(5, 2, i), (h // m_x, f // n_y), BF16, std=h ** -0.5) for i, k in enumerate(keys)}
    bufs = workloads.mlp_2d({k: v.cuda() for k, v in xb.items()}, {k: v.cuda() for k, v in w1.items()},
                            {k: v.cuda() for k, v in w2.items()}, m_x, n_y)
    coco.coco_device_status()
    ref = oracle.mlp_2d_forward({k: f64(v) for k, v in xb.items()}, {k: f64(v) for k, v in w1.items()},
                                {k: f64(v) for k, v in w2.items()}, m_x, n_y)
    for k in keys:
        # h is rounded to bf16 between the einsums on the GPU; the oracle keeps float64
        assert_close(bufs["y"][k], ref[k], BF16, f"device {k}")


# ------------------------------------------------------------------ full size


def cuda_gen(seed, shape, dtype, std=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.empty(shape, device="cuda").normal_(0.0, std, generator=g).to(dtype)


@pytest.mark.slow
def test_config2_full_size_sampled(coco, workloads):
    n, rows, hidden = 8, 8192, 4096
    ins = [cuda_gen(synth.seed_of(2, 0, r), (rows, hidden // n), F16) for r in range(n)]
    ws = [cuda_gen(synth.seed_of(2, 1, r), (hidden // n, hidden), F16, 0.02) for r in range(n)]
    bias = cuda_gen(synth.seed_of(2, 2), (hidden,), F16, 0.02)
    res = cuda_gen(synth.seed_of(2, 3), (rows, hidden), F16)
    _, out = workloads.megatron_attention_tail(ins, ws, bias, res, 0.1, 0)
    torch.cuda.synchronize()
    sel = np.unique(np.concatenate([[0, rows - 1], np.random.default_rng(2).choice(rows, 254, replace=False)]))
    idx = sel[:, None].astype(np.uint64) * np.uint64(hidden) + np.arange(hidden, dtype=np.uint64)[None, :]
    st = torch.from_numpy(sel).cuda()
    layers = [oracle.einsum("mk,kn->mn", f64(a[st]), f64(w)) for a, w in zip(ins, ws)]
    ref = oracle.fused_allreduce(layers, f64(bias), f64(res[st]), 0.1, 0, index=idx)
    for q, o in enumerate(out):
        assert_close(o[st], ref, F16, f"rank {q}")


@pytest.mark.slow
def test_config3_case1_full_size_sampled(coco):
    n, m, k, nn = 8, 16384, 8192, 3072
    a = [cuda_gen(synth.seed_of(3, 0, s), (m // n, k), BF16, k ** -0.5) for s in range(n)]
    b = [cuda_gen(synth.seed_of(3, 1, r), (k, nn), BF16) for r in range(n)]
    out = [torch.empty((m, nn), dtype=BF16, device="cuda") for _ in range(n)]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(a, 0), coco.local(b), coco.local(out))
    coco.coco_device_status()
    sel = np.unique(np.concatenate([[0, m // n - 1], np.random.default_rng(3).choice(m // n, 14, replace=False)]))
    st = torch.from_numpy(sel).cuda()
    refs = oracle.allgather_einsum("mk,kn->mn", "lhs", "m", [f64(x[st]) for x in a], [f64(x) for x in b])
    rows = torch.from_numpy(np.concatenate([s * (m // n) + sel for s in range(n)])).cuda()
    for r in range(n):
        assert_close(out[r][rows], refs[r], BF16, f"rank {r}")


@pytest.mark.slow
def test_config4a_case2_full_size_sampled(coco):
    n, m, k, nn = 8, 8192, 16384, 8192
    a = [cuda_gen(synth.seed_of(4, 0, s), (m, k // n), BF16) for s in range(n)]
    b = [cuda_gen(synth.seed_of(4, 1, r), (k, nn), BF16) for r in range(n)]
    out = [torch.empty((m, nn), dtype=F32, device="cuda") for _ in range(n)]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(a, 1), coco.local(b), coco.local(out))
    coco.coco_device_status()
    sel = np.unique(np.concatenate([[0, m - 1], np.random.default_rng(4).choice(m, 14, replace=False)]))
    st = torch.from_numpy(sel).cuda()
    for r in (0, 5):  # two ranks: each needs its own 16384 x 8192 local operand on the host
        ref = oracle.allgather_einsum("mk,kn->mn", "lhs", "k", [f64(x[st]) for x in a], [f64(b[r])])[0]
        # a bf16 configuration (bf16 inputs, fp32 accumulation and output): the 16-bit bar applies
        assert_close(out[r][st], ref, BF16, f"rank {r}")
        # outputs have magnitude ~sqrt(K) = 128; relative to that scale the fp32 sum is far tighter
        assert (np.abs(f64(out[r][st]) - ref) / (np.abs(ref) + np.sqrt(k))).max() < 1e-4


@pytest.mark.slow
def test_config4b_case3_full_size_sampled(coco):
    n, bt, m, k, nn = 8, 64, 1024, 128, 1024
    ls = [cuda_gen(synth.seed_of(4, 2, s), (bt // n, m, k), BF16) for s in range(n)]
    rs = [cuda_gen(synth.seed_of(4, 3, r), (bt, k, nn), BF16) for r in range(n)]
    out = [torch.empty((bt, m, nn), dtype=BF16, device="cuda") for _ in range(n)]
    coco.coco_looped_ag_einsum("bmk,bkn->bmn", coco.sliced(ls, 0), coco.local(rs), coco.local(out))
    coco.coco_device_status()
    js = [0, 3, 7]  # local batch indices sampled in every shard
    gb = torch.tensor([s * (bt // n) + j for s in range(n) for j in js], device="cuda")
    refs = oracle.allgather_einsum("bmk,bkn->bmn", "lhs", "b", [f64(x[js]) for x in ls], [f64(x[gb]) for x in rs])
    for r in range(n):
        assert_close(out[r][gb], refs[r], BF16, f"rank {r}")


@pytest.mark.slow
def test_config5_mesh_full_size_sampled(coco, workloads):
    m_x, n_y, b, f, h = 2, 4, 8192, 8192, 32768
    keys = [(x, y) for x in range(m_x) for y in range(n_y)]
    xb = {k: cuda_gen(synth.seed_of(5, 0, i), (b // n_y, f // m_x), BF16) for i, k in enumerate(keys)}
    w1 = {k: cuda_gen(synth.seed_of(5, 1, i), (f // n_y, h // m_x), BF16, f ** -0.5) for i, k in enumerate(keys)}
    w2 = {k: cuda_gen(synth.seed_of(5, 2, i), (h // m_x, f // n_y), BF16, h ** -0.5) for i, k in enumerate(keys)}
    bufs = workloads.mlp_2d(xb, w1, w2, m_x, n_y)
    coco.coco_device_status()
    sel = torch.tensor([0, 777, b // n_y - 1], device="cuda")
    ref = oracle.mlp_2d_forward({k: f64(v[sel]) for k, v in xb.items()}, {k: f64(v) for k, v in w1.items()},
                                {k: f64(v) for k, v in w2.items()}, m_x, n_y)
    for k in keys:
        assert_close(bufs["y"][k][sel], ref[k], BF16, f"device {k}")
    del bufs
    torch.cuda.empty_cache()
