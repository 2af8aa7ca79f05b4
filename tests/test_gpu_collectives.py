"""GPU parity of the reduction kernels against the oracle, through the C-ABI.

FusedAllReduce, AllReduce, ReduceScatter, AllGather and AllReduce Split RS-AG
([CoCoNet] §5.2 and the split transformation; [Decomp] §2.1). Masks are
compared bit for bit, AllGather and RS-AG vs AllReduce are bit-exact, the rest
within |gpu - ref| <= tol * (|ref| + 1) with tol 1e-5 (fp32) / 2e-2 (16-bit).
"""

import numpy as np
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


DTYPES = [torch.float32, torch.float16, torch.bfloat16]


def run_far(coco, n, shape, dtype, bias=True, res=True, p=0.1, seed=7, cfg=1, out_aliased=False):
    parts = synth.per_rank(cfg, 0, n, shape, dtype, "uniform")
    b = synth.tensor(synth.seed_of(cfg, 1), (shape[-1],), dtype, "uniform") if bias else None
    r = synth.tensor(synth.seed_of(cfg, 2), shape, dtype, "uniform") if res else None
    if out_aliased:
        one = empty_like_list(1, shape, dtype)[0]
        outs = [one] * n
    else:
        outs = empty_like_list(n, shape, dtype)
    coco.coco_fused_allreduce(coco.local(dev(parts)), None if b is None else b.cuda(),
                              None if r is None else coco.replicated([r.cuda()] * n), p, seed,
                              coco.replicated(outs))
    torch.cuda.synchronize()
    ref = oracle.fused_allreduce([f64(x) for x in parts], None if b is None else f64(b),
                                 None if r is None else f64(r), p, seed)
    return outs, ref, r


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 8, 11])
@pytest.mark.parametrize("shape", [(4, 16), (37, 24), (3, 129, 64)])
def test_fused_allreduce_matches_oracle(coco, dtype, n, shape):
    outs, ref, _ = run_far(coco, n, shape, dtype)
    for q, o in enumerate(outs):
        assert_close(o, ref, dtype, f"rank {q}")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])  # replicated: bitwise identical on every rank


@pytest.mark.parametrize("dtype", DTYPES)
def test_fused_allreduce_at_row_chunks_equal_the_whole_call(coco, dtype):
    """[CoCoNet] §5.3 Overlap in chunks: FusedAllReduce over consecutive row ranges with the ranges'
    whole-tensor index bases gives, bit for bit, the one-call result (dropout mask included)."""
    n, rows, h, p, seed = 4, 40, 64, 0.3, 77
    parts = dev(synth.per_rank(31, 0, n, (rows, h), dtype, "uniform"))
    b = synth.tensor(synth.seed_of(31, 1), (h,), dtype, "uniform").cuda()
    r = synth.tensor(synth.seed_of(31, 2), (rows, h), dtype, "uniform").cuda()
    whole = empty_like_list(n, (rows, h), dtype)
    coco.coco_fused_allreduce(coco.local(parts), b, coco.replicated([r] * n), p, seed, coco.replicated(whole))
    chunked = empty_like_list(n, (rows, h), dtype)
    for r0, r1 in [(0, 8), (8, 24), (24, 40)]:
        coco.coco_fused_allreduce_at(coco.local([x[r0:r1] for x in parts]), b, coco.replicated([r[r0:r1]] * n), p,
                                     seed, r0 * h, coco.replicated([o[r0:r1] for o in chunked]))
    torch.cuda.synchronize()
    for q in range(n):
        assert torch.equal(chunked[q], whole[q])
    ref = oracle.fused_allreduce([f64(x) for x in parts], f64(b), f64(r), p, seed)
    assert_close(chunked[0], ref, dtype, "chunked")


@pytest.mark.parametrize("dtype", DTYPES)
def test_fused_allreduce_at_keeps_the_bias_phase_off_a_row_boundary(coco, dtype):
    """A part that starts mid-row (index_base not a multiple of the row length) still takes bias
    element (e mod H) and dropout index e of the whole tensor."""
    n, rows, h, p, seed, off, m = 3, 16, 64, 0.2, 5, 8, 4
    parts = dev(synth.per_rank(32, 0, n, (rows, h), dtype, "uniform"))
    b = synth.tensor(synth.seed_of(32, 1), (h,), dtype, "uniform").cuda()
    r = synth.tensor(synth.seed_of(32, 2), (rows, h), dtype, "uniform").cuda()
    whole = empty_like_list(n, (rows, h), dtype)
    coco.coco_fused_allreduce(coco.local(parts), b, coco.replicated([r] * n), p, seed, coco.replicated(whole))

    def part(t):
        return t.reshape(-1)[off:off + m * h].view(m, h)

    outs = empty_like_list(n, (m, h), dtype)
    coco.coco_fused_allreduce_at(coco.local([part(x) for x in parts]), b, coco.replicated([part(r)] * n), p, seed,
                                 off, coco.replicated(outs))
    torch.cuda.synchronize()
    for q in range(n):
        assert torch.equal(outs[q], part(whole[q]))
    ref = oracle.fused_allreduce([f64(x) for x in parts], f64(b), f64(r), p, seed).reshape(-1)[off:off + m * h]
    assert_close(outs[0], ref.reshape(m, h), dtype, "mid-row part")


@pytest.mark.parametrize("bias,res,p", [(False, False, 0.0), (True, False, 0.0), (False, True, 0.5),
                                        (True, True, 0.0), (False, False, 0.3), (True, True, 1.0)])
def test_fused_allreduce_optional_parts(coco, bias, res, p):
    outs, ref, _ = run_far(coco, 4, (64, 128), torch.float32, bias, res, p)
    for o in outs:
        assert_close(o, ref, torch.float32)


def test_config1_fused_allreduce(coco):
    # 2 ranks, fp32 U(-1,1), local [4,16] + bias[16] + dropout p=0.1 (seed 0) + replicated residual [4,16]
    outs, ref, _ = run_far(coco, 2, (4, 16), torch.float32, True, True, 0.1, seed=0, cfg=1)
    for o in outs:
        assert_close(o, ref, torch.float32)


@pytest.mark.parametrize("dtype", DTYPES)
def test_dropped_elements_are_exactly_the_residual(coco, dtype):
    shape, p, seed = (256, 512), 0.25, 99
    outs, _, r = run_far(coco, 3, shape, dtype, True, True, p, seed)
    keep = oracle.keep_mask(seed, p, np.arange(np.prod(shape))).reshape(shape)
    got = outs[0].cpu()
    assert (~keep).sum() > 0
    assert torch.equal(got[torch.from_numpy(~keep)], r[torch.from_numpy(~keep)])


@pytest.mark.parametrize("seed,p,first", [(0, 0.1, 0), (1234567, 0.5, 12345), (2**63 + 11, 0.9, 2**40 - 7),
                                          (5, 0.0, 0), (5, 1.0, 0), (77, 0.3, 2**62)])
def test_keep_mask_bit_exact(coco, seed, p, first):
    count = (1 << 20) + 3
    mask = torch.empty(count, dtype=torch.uint8, device="cuda")
    coco.coco_dropout_keep_mask(seed, p, first, count, mask)
    torch.cuda.synchronize()
    want = oracle.keep_mask(seed, p, np.arange(count, dtype=np.uint64) + np.uint64(first))
    assert np.array_equal(mask.cpu().numpy().astype(bool), want)


def test_fused_allreduce_aliased_output_and_in_place(coco):
    outs, ref, _ = run_far(coco, 4, (32, 64), torch.bfloat16, out_aliased=True)
    assert_close(outs[0], ref, torch.bfloat16)
    # in place: out_q is partials_q
    n, shape = 4, (33, 64)
    parts = dev(synth.per_rank(3, 0, n, shape, torch.float16, "uniform"))
    ref = oracle.fused_allreduce([f64(x) for x in parts])
    coco.coco_allreduce(coco.local(parts), coco.replicated(parts))
    torch.cuda.synchronize()
    for x in parts:
        assert_close(x, ref, torch.float16)


def test_fused_allreduce_groups(coco):
    g, n, shape = 3, 2, (16, 32)
    parts = synth.per_rank(4, 0, g * n, shape, torch.float32, "uniform")
    outs = empty_like_list(g * n, shape, torch.float32)
    bias = synth.tensor(5, (32,), torch.float32, "uniform")
    coco.coco_fused_allreduce(coco.local(dev(parts), ngroups=g), bias.cuda(), None, 0.2, 3,
                              coco.replicated(outs, ngroups=g))
    torch.cuda.synchronize()
    for gi in range(g):
        ref = oracle.fused_allreduce([f64(x) for x in parts[gi * n:(gi + 1) * n]], f64(bias), None, 0.2, 3)
        for q in range(n):
            assert_close(outs[gi * n + q], ref, torch.float32, f"group {gi} rank {q}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n,shape,dim", [(2, (16, 24), 0), (4, (8, 64), 1), (8, (64, 40), 0), (3, (6, 9, 16), 1),
                                         (5, (2, 3, 80), 2), (1, (8, 8), 0)])
def test_reduce_scatter_and_allgather(coco, dtype, n, shape, dim):
    ins = synth.per_rank(6, 0, n, shape, dtype, "uniform")
    sl_shape = list(shape)
    sl_shape[dim] //= n
    scat = empty_like_list(n, sl_shape, dtype)
    coco.coco_reduce_scatter(coco.local(dev(ins)), coco.sliced(scat, dim))
    torch.cuda.synchronize()
    ref = oracle.reduce_scatter([f64(x) for x in ins], dim)
    for r in range(n):
        assert_close(scat[r], ref[r], dtype, f"reduce-scatter rank {r}")
    # all-gather of the (rounded) slices is a bit-exact concatenation
    outs = empty_like_list(n, shape, dtype)
    coco.coco_allgather(coco.sliced(scat, dim), coco.replicated(outs))
    torch.cuda.synchronize()
    want = torch.cat([s.cpu() for s in scat], dim)
    for o in outs:
        assert torch.equal(o.cpu(), want)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n,shape,dim", [(8, (4096,), 0), (4, (64, 96), 1), (3, (9, 40), 0), (8, (16, 8, 64), 1)])
def test_allreduce_split_rs_ag_is_bit_identical_to_allreduce(coco, dtype, n, shape, dim):
    ins = dev(synth.per_rank(7, 0, n, shape, dtype, "uniform"))
    sl = list(shape)
    sl[dim] //= n
    scratch = empty_like_list(n, sl, dtype)
    split = empty_like_list(n, shape, dtype)
    direct = empty_like_list(n, shape, dtype)
    coco.coco_allreduce_rs_ag(coco.local(ins), coco.sliced(scratch, dim), coco.replicated(split))
    coco.coco_allreduce(coco.local(ins), coco.replicated(direct))
    torch.cuda.synchronize()
    ref = oracle.allreduce_split_rs_ag([f64(x) for x in ins], dim)[0]
    for a, b in zip(split, direct):
        assert torch.equal(a, b)
        assert_close(a, ref, dtype)


def test_empty_and_degenerate(coco):
    z = [torch.empty((0, 16), device="cuda") for _ in range(2)]
    coco.coco_fused_allreduce(coco.local(z), None, None, 0.5, 1, coco.replicated(z))
    one = dev(synth.per_rank(8, 0, 1, (5, 8), torch.float32, "uniform"))
    out = empty_like_list(1, (5, 8), torch.float32)
    coco.coco_allreduce(coco.local(one), coco.replicated(out))
    torch.cuda.synchronize()
    assert torch.equal(out[0], one[0])  # N = 1: the identity


@pytest.mark.slow
def test_config2_fused_allreduce_full_size_sampled(coco):
    """N=8 fp16 [8*1024, 4096] partials + bias + p=0.1 + residual, in the launch
    configuration the bench uses; the oracle checks 1024 sampled rows plus the
    first and last rows, with their global element indices."""
    n, rows, h = 8, 8192, 4096
    parts = synth.per_rank(2, 0, n, (rows, h), torch.float16, "normal", 0.45)
    bias = synth.tensor(synth.seed_of(2, 1), (h,), torch.float16, "normal", 0.02)
    res = synth.tensor(synth.seed_of(2, 2), (rows, h), torch.float16)
    outs = empty_like_list(n, (rows, h), torch.float16)
    coco.coco_fused_allreduce(coco.local(dev(parts)), bias.cuda(), coco.replicated([res.cuda()] * n), 0.1, 0,
                              coco.replicated(outs))
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    sample = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 1024, replace=False)]))
    idx = sample[:, None].astype(np.uint64) * np.uint64(h) + np.arange(h, dtype=np.uint64)[None, :]
    ref = oracle.fused_allreduce([f64(x[sample]) for x in parts], f64(bias), f64(res[sample]), 0.1, 0, index=idx)
    for q in range(n):
        assert_close(outs[q].cpu()[sample], ref, torch.float16, f"rank {q}")


@pytest.mark.slow
def test_config5b_allreduce_rs_ag_full_size(coco):
    """1 GiB fp32 per rank over N=8: RS-AG bit-identical to the direct AllReduce,
    and sampled elements within 1e-5 of the oracle."""
    n, numel = 8, 1 << 28
    ins = [torch.empty(numel, device="cuda") for _ in range(n)]
    g = torch.Generator(device="cuda")
    for r, x in enumerate(ins):
        g.manual_seed(synth.seed_of(5, 0, r))
        x.uniform_(-1, 1, generator=g)
    scratch = [torch.empty(numel // n, device="cuda") for _ in range(n)]
    outs = [torch.empty(numel, device="cuda") for _ in range(n)]
    coco.coco_allreduce_rs_ag(coco.local(ins), coco.sliced(scratch, 0), coco.replicated(outs))
    direct = torch.empty(numel, device="cuda")
    coco.coco_allreduce(coco.local(ins), coco.replicated([direct] * n))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, direct)
    idx = torch.from_numpy(np.random.default_rng(1).choice(numel, 1 << 16, replace=False)).cuda()
    ref = oracle.allreduce([f64(x[idx]) for x in ins])[0]
    assert_close(direct[idx], ref, torch.float32)
    del ins, outs, scratch
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n,g", [(64, 1), (16, 4), (9, 7)])
def test_at_the_pointer_limit(coco, n, g):
    """nranks x ngroups up to the interface's 64 pointers: FusedAllReduce (the runtime rank-count path,
    8 ranks at a time), ReduceScatter and AllGather."""
    dtype, shape = torch.float16, (8, 64)
    parts = dev(synth.per_rank(33, 0, n * g, shape, dtype, "uniform"))
    bias = synth.tensor(synth.seed_of(33, 1), (64,), dtype, "uniform").cuda()
    outs = empty_like_list(n * g, shape, dtype)
    coco.coco_fused_allreduce(coco.local(parts, ngroups=g), bias, None, 0.25, 11, coco.replicated(outs, ngroups=g))
    torch.cuda.synchronize()
    for gi in range(g):
        ref = oracle.fused_allreduce([f64(x) for x in parts[gi * n:(gi + 1) * n]], f64(bias), None, 0.25, 11)
        for q in range(n):
            assert_close(outs[gi * n + q], ref, dtype, f"group {gi} rank {q}")
    rs_shape = (n * 2, 16)
    ins = dev(synth.per_rank(34, 0, n * g, rs_shape, torch.float32, "uniform"))
    scat = empty_like_list(n * g, (2, 16), torch.float32)
    coco.coco_reduce_scatter(coco.local(ins, ngroups=g), coco.sliced(scat, 0, ngroups=g))
    full = empty_like_list(n * g, rs_shape, torch.float32)
    coco.coco_allgather(coco.sliced(scat, 0, ngroups=g), coco.replicated(full, ngroups=g))
    torch.cuda.synchronize()
    for gi in range(g):
        ref = oracle.reduce_scatter([f64(x) for x in ins[gi * n:(gi + 1) * n]], 0)
        for r in range(n):
            assert_close(scat[gi * n + r], ref[r], torch.float32, f"group {gi} slice {r}")
        want = torch.cat([s.cpu() for s in scat[gi * n:(gi + 1) * n]], 0)
        for q in range(n):
            assert torch.equal(full[gi * n + q].cpu(), want)


@pytest.mark.slow
def test_fused_allreduce_beyond_32_bit_element_indices(coco):
    """A tensor of 2^31 + 4096 fp16 elements per rank (4 GiB): element offsets, dropout indices and
    the bias phase past 2^31 are 64-bit. Sampled rows near the start, across the 2^31 boundary and at
    the end match the oracle evaluated at their whole-tensor indices; the mask there is bit-exact."""
    n, h = 2, 4096
    rows = (1 << 31) // h + 1
    g = torch.Generator(device="cuda")
    parts = []
    for r in range(n):
        x = torch.empty((rows, h), dtype=torch.float16, device="cuda")
        g.manual_seed(synth.seed_of(36, 0, r))
        x.uniform_(-1, 1, generator=g)
        parts.append(x)
    bias = synth.tensor(synth.seed_of(36, 1), (h,), torch.float16, "uniform").cuda()
    res = torch.empty((rows, h), dtype=torch.float16, device="cuda")
    g.manual_seed(synth.seed_of(36, 2))
    res.uniform_(-1, 1, generator=g)
    out = torch.empty((rows, h), dtype=torch.float16, device="cuda")
    coco.coco_fused_allreduce(coco.local(parts), bias, coco.replicated([res] * n), 0.5, 99, coco.replicated([out] * n))
    coco.coco_device_status()
    sample = np.array([0, 1, rows // 2, rows - 3, rows - 2, rows - 1])
    idx = sample[:, None].astype(np.uint64) * np.uint64(h) + np.arange(h, dtype=np.uint64)[None, :]
    assert int(idx.max()) >= (1 << 31)
    ref = oracle.fused_allreduce([f64(x[sample]) for x in parts], f64(bias), f64(res[sample]), 0.5, 99, index=idx)
    got = out[torch.from_numpy(sample).cuda()]
    assert_close(got, ref, torch.float16, "rows past 2^31")
    keep = oracle.keep_mask(99, 0.5, idx.ravel()).reshape(idx.shape)
    dropped = torch.from_numpy(~keep).cuda()
    assert torch.equal(got[dropped], res[torch.from_numpy(sample).cuda()][dropped])
    del parts, res, out
