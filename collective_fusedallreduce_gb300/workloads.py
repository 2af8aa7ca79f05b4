"""The pages' composite workloads as sequences of C-ABI calls.

Each function only allocates output buffers (PyTorch) and orders calls into
libcoco; every arithmetic step runs in the library's kernels.

* ``megatron_attention_tail``: [CoCoNet] Fig. 3 -- the local MatMul of two
  tensors sliced on the contracting dimension, then FusedAllReduce with bias,
  dropout and residual.
* ``megatron_attention_tail_overlap``: the same with [CoCoNet] §5.3's Overlap
  construct in row chunks (FusedAllReduce of one chunk beside the MatMul of
  the next, on two streams).
* ``mlp_1d``: the 1-D partitioned two-layer MLP of [Decomp] §2.2 Fig. 2
  (Looped AllGather-Einsum case 1, then Looped Einsum-ReduceScatter).
* ``mlp_2d``: the [M, N]-mesh two-layer MLP of [Decomp] §2.2 Fig. 3:
  AllGather of X along x, Looped AllGather-Einsum of W1 along y (contracting
  dimension, Addition), AllGather of W2 along y, Looped Einsum-ReduceScatter
  along x (the subgroup ReduceScatter of the figure).
"""

import torch

from . import coco


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def megatron_attention_tail(in_slices, w_slices, bias, residual, p, seed, layer=None, out=None, stream=None):
    """``layer_r = in_r @ w_r`` (local), then ``out = FusedAllReduce(layer) + b -> dropout -> + residual``.

    ``in_slices[r]``: [rows, H/N] (slice r of ``in`` on its last dimension);
    ``w_slices[r]``: [H/N, H] (slice r of ``w`` on its first); ``residual``:
    one [rows, H] tensor (replicated). ``layer`` / ``out``: optional
    preallocated per-rank buffers. Returns (layer, out).
    """
    n = len(in_slices)
    rows, h = in_slices[0].shape[0], w_slices[0].shape[1]
    dt, dev = in_slices[0].dtype, in_slices[0].device
    layer = layer if layer is not None else [_empty((rows, h), dt, dev) for _ in range(n)]
    out = out if out is not None else [_empty((rows, h), dt, dev) for _ in range(n)]
    coco.coco_einsum("mk,kn->mn", coco.sliced(in_slices, 1), coco.sliced(w_slices, 0), coco.local(layer), stream)
    coco.coco_fused_allreduce(coco.local(layer), bias, None if residual is None else coco.replicated([residual] * n),
                              p, seed, coco.replicated(out), stream)
    return layer, out


def megatron_attention_tail_overlap(in_slices, w_slices, bias, residual, p, seed, chunks, layer=None, out=None,
                                    stream=None, side_stream=None):
    """The same tail with [CoCoNet] §5.3's Overlap construct, in chunks: the rows are cut into
    ``chunks`` ranges; the MatMul of each range runs on ``stream`` and its FusedAllReduce on
    ``side_stream`` as soon as that range's partials exist, so the FusedAllReduce of one range runs
    while the MatMul computes the next. Ordering is by CUDA events only (nothing waits on the device).
    The FusedAllReduce of a range passes the range's whole-tensor index base, so the result equals
    ``megatron_attention_tail``'s bit for bit. ``stream`` waits for the last FusedAllReduce before
    returning. Returns (layer, out)."""
    n = len(in_slices)
    rows, h = in_slices[0].shape[0], w_slices[0].shape[1]
    dt, dev = in_slices[0].dtype, in_slices[0].device
    layer = layer if layer is not None else [_empty((rows, h), dt, dev) for _ in range(n)]
    out = out if out is not None else [_empty((rows, h), dt, dev) for _ in range(n)]
    main = stream if stream is not None else torch.cuda.current_stream(dev)
    side = side_stream if side_stream is not None else torch.cuda.Stream(device=dev)
    chunks = max(1, min(int(chunks), rows))
    bounds = [rows * c // chunks for c in range(chunks + 1)]
    for r0, r1 in zip(bounds[:-1], bounds[1:]):
        if r1 == r0:
            continue
        coco.coco_einsum("mk,kn->mn", coco.sliced([x[r0:r1] for x in in_slices], 1), coco.sliced(w_slices, 0),
                         coco.local([x[r0:r1] for x in layer]), main)
        ready = torch.cuda.Event()
        ready.record(main)
        side.wait_event(ready)
        coco.coco_fused_allreduce_at(coco.local([x[r0:r1] for x in layer]), bias,
                                     None if residual is None else coco.replicated([residual[r0:r1]] * n),
                                     p, seed, r0 * h, coco.replicated([x[r0:r1] for x in out]), side)
    done = torch.cuda.Event()
    done.record(side)
    main.wait_event(done)
    return layer, out


def mlp_1d(x_shards, w1_cols, w2_rows, h=None, y=None, stream=None):
    """Fig. 2 forward: ``h_r = AllGather(x) @ W1_r`` (case 1, looped over the
    batch shards), then ``y = ReduceScatter(h_r @ W2_r)`` over the batch
    dimension (looped). Returns (h, y)."""
    n = len(x_shards)
    b, f = x_shards[0].shape[0] * n, x_shards[0].shape[1]
    hn = w1_cols[0].shape[1]
    dt, dev = x_shards[0].dtype, x_shards[0].device
    h = h if h is not None else [_empty((b, hn), dt, dev) for _ in range(n)]
    y = y if y is not None else [_empty((b // n, f), dt, dev) for _ in range(n)]
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.sliced(x_shards, 0), coco.local(w1_cols), coco.local(h), stream)
    coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(h, 1), coco.sliced(w2_rows, 0), coco.sliced(y, 0), stream)
    return h, y


def mesh_order(blocks, m_x, n_y, group_axis):
    """Group-major list of per-device tensors: ``group_axis="y"`` gives groups of
    fixed y (ranks along x), ``"x"`` groups of fixed x (ranks along y)."""
    if group_axis == "y":
        return [blocks[(x, y)] for y in range(n_y) for x in range(m_x)]
    return [blocks[(x, y)] for x in range(m_x) for y in range(n_y)]


def mlp_2d(x_blocks, w1_blocks, w2_blocks, m_x, n_y, bufs=None, stream=None, side_stream=None):
    """Two-layer MLP on an [M, N] device mesh; device (x, y) holds
    X(x,y) = [B/N, F/M], W1(x,y) = [F/N, H/M], W2(x,y) = [H/M, F/N] (dicts
    keyed by (x, y)). Returns a dict of intermediate and output buffers keyed
    "xf", "h", "w2f", "y" (each a dict keyed by (x, y)).

    With ``side_stream``, the AllGather of W2 (independent of the first einsum)
    runs on it beside the first einsum, ordered by events: it starts once the
    AllGather of X is done (so the einsum's persistent kernel is placed on the
    SMs with it) and the Einsum-ReduceScatter waits for it. The results are the
    same bits as the one-stream order.
    """
    keys = [(x, y) for x in range(m_x) for y in range(n_y)]
    bt, fm = x_blocks[(0, 0)].shape
    fn, hm = w1_blocks[(0, 0)].shape
    dt, dev = x_blocks[(0, 0)].dtype, x_blocks[(0, 0)].device
    f = fm * m_x
    if bufs is None:
        bufs = {
            "xf": {k: _empty((bt, f), dt, dev) for k in keys},
            "h": {k: _empty((bt, hm), dt, dev) for k in keys},
            "w2f": {k: _empty((hm, f), dt, dev) for k in keys},
            "y": {k: _empty((bt, fm), dt, dev) for k in keys},
        }
    main = stream if stream is not None else torch.cuda.current_stream(dev)
    # 1. AllGather X along x (subgroups of fixed y), on X's feature dimension
    coco.coco_allgather(coco.sliced(mesh_order(x_blocks, m_x, n_y, "y"), 1, ngroups=n_y),
                        coco.replicated(mesh_order(bufs["xf"], m_x, n_y, "y"), ngroups=n_y), main)
    w2_stream = main
    if side_stream is not None:
        after_x = torch.cuda.Event()
        after_x.record(main)  # also orders it after the previous call's reads of W2's gather
        side_stream.wait_event(after_x)
        w2_stream = side_stream
    # 2. Looped AllGather-Einsum of W1 along y (subgroups of fixed x), case 2 with the looped operand on the right
    coco.coco_looped_ag_einsum("mk,kn->mn", coco.local(mesh_order(bufs["xf"], m_x, n_y, "x"), ngroups=m_x),
                               coco.sliced(mesh_order(w1_blocks, m_x, n_y, "x"), 0, ngroups=m_x),
                               coco.local(mesh_order(bufs["h"], m_x, n_y, "x"), ngroups=m_x), main)
    # 3. AllGather W2 along y (subgroups of fixed x), on W2's feature dimension
    coco.coco_allgather(coco.sliced(mesh_order(w2_blocks, m_x, n_y, "x"), 1, ngroups=m_x),
                        coco.replicated(mesh_order(bufs["w2f"], m_x, n_y, "x"), ngroups=m_x), w2_stream)
    if w2_stream is not main:
        w2_done = torch.cuda.Event()
        w2_done.record(w2_stream)
        main.wait_event(w2_done)
    # 4. Looped Einsum-ReduceScatter along x (subgroups of fixed y) onto the feature dimension
    coco.coco_looped_einsum_rs("mk,kn->mn", coco.sliced(mesh_order(bufs["h"], m_x, n_y, "y"), 1, ngroups=n_y),
                               coco.sliced(mesh_order(bufs["w2f"], m_x, n_y, "y"), 0, ngroups=n_y),
                               coco.sliced(mesh_order(bufs["y"], m_x, n_y, "y"), 1, ngroups=n_y), main)
    return bufs
