"""GPU parity of coco_matmul_fused_allreduce: the local MatMul of [CoCoNet] Fig. 3
fused with its FusedAllReduce (bias, dropout, residual) in one tensor-core kernel.

Compared with the oracle's unfused chain (per-rank partials in float64, summed in
rank order, then bias, dropout, residual), element by element within the 16-bit
bar, with the dropout decisions checked bit for bit through the dropped elements.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_fusedallreduce_gb300 import synth
from helpers import assert_close, dev, f64

pytestmark = pytest.mark.gpu

BF16, F16 = torch.bfloat16, torch.float16


@pytest.fixture(scope="module")
def coco():
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import coco as c
    return c


def run(coco, n, m, ks, nn, dtype, bias=True, res=True, p=0.1, seed=3, ngroups=1, cfg=20):
    ins = synth.per_rank(cfg, 0, n * ngroups, (m, ks), dtype)
    ws = synth.per_rank(cfg, 1, n * ngroups, (ks, nn), dtype, std=(n * ks) ** -0.5)
    b = synth.tensor(synth.seed_of(cfg, 2), (nn,), dtype, std=0.5) if bias else None
    rs = [synth.tensor(synth.seed_of(cfg, 3, g), (m, nn), dtype) for g in range(ngroups)] if res else None
    outs = [torch.full((m, nn), float("nan"), dtype=dtype, device="cuda") for _ in range(n * ngroups)]
    rdev = [r.cuda() for r in rs] if res else None
    coco.coco_matmul_fused_allreduce(
        "mk,kn->mn", coco.sliced(dev(ins), 1, ngroups), coco.sliced(dev(ws), 0, ngroups),
        None if b is None else b.cuda(),
        None if rs is None else coco.replicated([rdev[g] for g in range(ngroups) for _ in range(n)], ngroups),
        p, seed, coco.replicated(outs, ngroups))
    coco.coco_device_status()
    refs = []
    for g in range(ngroups):
        sl = slice(g * n, (g + 1) * n)
        _, ref = oracle.megatron_attention_tail([f64(x) for x in ins[sl]], [f64(w) for w in ws[sl]],
                                                None if b is None else f64(b), None if rs is None else f64(rs[g]),
                                                p, seed)
        refs.append(ref)
    return outs, refs, rs


@pytest.mark.parametrize("dtype", [F16, BF16])
# (column counts: 520, 264, 136 are not whole 64-column blocks, 256 / 320 / 192 are: an even and two odd
# numbers of blocks for the two-strip stores of the pair-MMA kernel)
@pytest.mark.parametrize("n,m,ks,nn", [(8, 264, 64, 520), (2, 128, 40, 256), (1, 136, 200, 264), (4, 300, 72, 136),
                                       (4, 264, 64, 320), (8, 136, 32, 192), (4, 256, 128, 256)])
def test_matches_oracle(coco, dtype, n, m, ks, nn):
    outs, refs, _ = run(coco, n, m, ks, nn, dtype)
    for q, o in enumerate(outs):
        assert_close(o, refs[0], dtype, f"replica {q}")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("bias,res,p", [(False, False, 0.0), (True, False, 0.0), (False, True, 0.5), (True, True, 1.0)])
def test_optional_parts(coco, bias, res, p):
    outs, refs, _ = run(coco, 4, 256, 64, 512, BF16, bias, res, p)
    for o in outs:
        assert_close(o, refs[0], BF16)


def test_dropped_elements_are_exactly_the_residual(coco):
    m, nn, p, seed = 256, 512, 0.3, 77
    outs, _, rs = run(coco, 4, m, 64, nn, F16, True, True, p, seed)
    keep = torch.from_numpy(oracle.keep_mask(seed, p, np.arange(m * nn)).reshape(m, nn))
    assert (~keep).sum() > 0
    assert torch.equal(outs[0].cpu()[~keep], rs[0][~keep])


def test_groups(coco):
    outs, refs, _ = run(coco, 2, 128, 64, 256, BF16, ngroups=3)
    for g in range(3):
        for q in range(2):
            assert_close(outs[g * 2 + q], refs[g], BF16, f"group {g} replica {q}")


def test_single_output_copy_and_residual_in_place(coco):
    n, m, ks, nn = 4, 128, 64, 256
    ins = dev(synth.per_rank(21, 0, n, (m, ks), BF16))
    ws = dev(synth.per_rank(21, 1, n, (ks, nn), BF16, std=0.1))
    r = synth.tensor(synth.seed_of(21, 3), (m, nn), BF16).cuda()
    ref = oracle.megatron_attention_tail([f64(x) for x in ins], [f64(w) for w in ws], None, f64(r), 0.2, 9)[1]
    coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(ins, 1), coco.sliced(ws, 0), None,
                                     coco.replicated([r] * n), 0.2, 9, coco.replicated([r] * n))
    coco.coco_device_status()
    assert_close(r, ref, BF16, "in place over the residual")


def test_rejections(coco):
    n = 2
    a = dev(synth.per_rank(22, 0, n, (64, 64), BF16))
    w = dev(synth.per_rank(22, 1, n, (64, 128), BF16))
    o = [torch.empty((64, 128), dtype=BF16, device="cuda") for _ in range(n)]
    with pytest.raises(coco.CocoError) as e:
        coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.local(a), coco.sliced(w, 0), None, None, 0.0, 0,
                                         coco.replicated(o))
    assert e.value.name == "COCO_ERR_LAYOUT"
    big = torch.empty((2, 64, 128), dtype=BF16, device="cuda")
    with pytest.raises(coco.CocoError) as e:  # one buffer used as a replica by two groups
        coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(a, 1, 2), coco.sliced(w, 0, 2), None, None, 0.0,
                                         0, coco.replicated([big[0], big[0]], 2))
    assert e.value.name == "COCO_ERR_ALIAS"
    f = [torch.empty((64, 128), dtype=torch.float32, device="cuda") for _ in range(n)]
    with pytest.raises(coco.CocoError) as e:
        coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(a, 1), coco.sliced(w, 0), None, None, 0.0, 0,
                                         coco.replicated(f))
    assert e.value.name in ("COCO_ERR_UNSUPPORTED", "COCO_ERR_DTYPE")


@pytest.mark.slow
def test_config2_fused_full_size_sampled(coco):
    """N=8 fp16, in[8,1024,4096] sliced on dim 2, w[4096,4096] sliced on dim 0, bias, p=0.1, residual."""
    n, rows, hidden = 8, 8192, 4096

    def g(seed, shape, std=1.0):
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        return torch.empty(shape, device="cuda").normal_(0.0, std, generator=gen).half()

    ins = [g(synth.seed_of(2, 0, r), (rows, hidden // n)) for r in range(n)]
    ws = [g(synth.seed_of(2, 1, r), (hidden // n, hidden), 0.02) for r in range(n)]
    bias = g(synth.seed_of(2, 2), (hidden,), 0.02)
    res = g(synth.seed_of(2, 3), (rows, hidden))
    outs = [torch.empty((rows, hidden), dtype=F16, device="cuda") for _ in range(n)]
    coco.coco_matmul_fused_allreduce("mk,kn->mn", coco.sliced(ins, 1), coco.sliced(ws, 0), bias,
                                     coco.replicated([res] * n), 0.1, 0, coco.replicated(outs))
    coco.coco_device_status()
    sel = np.unique(np.concatenate([[0, rows - 1], np.random.default_rng(9).choice(rows, 254, replace=False)]))
    st = torch.from_numpy(sel).cuda()
    idx = sel[:, None].astype(np.uint64) * np.uint64(hidden) + np.arange(hidden, dtype=np.uint64)[None, :]
    layers = [oracle.einsum("mk,kn->mn", f64(a[st]), f64(w)) for a, w in zip(ins, ws)]
    ref = oracle.fused_allreduce(layers, f64(bias), f64(res[st]), 0.1, 0, index=idx)
    for q, o in enumerate(outs):
        assert_close(o[st], ref, F16, f"replica {q}")
