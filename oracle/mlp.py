"""Composite workloads built from the collectives (test infrastructure only).

* ``mlp_1d_forward``: the two-layer MLP of [Decomp] §2.2 Fig. 2, N-way 1-D
  partitioned, activations kept sharded on the batch dimension.
* ``mlp_2d_forward``: the two-layer MLP of [Decomp] §2.2 Fig. 3 on a logical
  [M, N] device mesh.
* ``megatron_attention_tail``: [CoCoNet] Fig. 3, MatMul of two sliced tensors
  (a local partial), then FusedAllReduce with bias, dropout and residual.

Each has a ``*_reference`` (or special-case) form computed without any
partitioning, which the tests use to pin the partitioned forms.
"""

import numpy as np

from .collectives import allgather
from .looped import (
    allgather_einsum,
    looped_allgather_einsum,
    einsum_reduce_scatter,
    looped_einsum_reduce_scatter,
)
from .fused import fused_allreduce
from .einsum import einsum


def mlp_1d_reference(x_full, w1_full, w2_full):
    """Unpartitioned y = (x @ W1) @ W2 (no activation: the pages name none)."""
    return einsum("mk,kn->mn", einsum("mk,kn->mn", x_full, w1_full), w2_full)


def mlp_1d_forward(x_shards, w1_parts, w2_parts, reading="megatron", looped=True):
    """N-way 1-D partitioned MLP forward ([Decomp] §2.2, Fig. 2).

    ``x_shards[r]``: rank r's batch shard of the activations, [B/N, F].

    ``reading="megatron"`` (the one the hot path runs): ``w1_parts[r]`` is
    column shard r of W1, [F, H/N]; ``w2_parts[r]`` is row shard r of W2,
    [H/N, F]. Einsum 1 is a Looped AllGather-Einsum of x over the batch
    dimension (case 1); einsum 2 is a Looped Einsum-ReduceScatter over the
    batch dimension of the output. Result: ``y_r`` = batch shard r, [B/N, F].

    ``reading="weights_gathered"`` (Fig. 2 taken literally): ``w1_parts[r]`` and
    ``w2_parts[r]`` are dim-0 shards of W1 [F, H] and W2 [H, F]; each einsum is
    a Looped AllGather-Einsum of the weight over its contracting dimension
    (case 2 with the looped operand on the right). Same result.

    ``looped=False`` uses the monolithic collective + einsum forms instead.
    """
    n = len(x_shards)
    ag = looped_allgather_einsum if looped else allgather_einsum
    rs = looped_einsum_reduce_scatter if looped else einsum_reduce_scatter
    if reading == "megatron":
        h = ag("mk,kn->mn", "lhs", "m", x_shards, w1_parts)
        return rs("mk,kn->mn", h, w2_parts, "m")
    if reading == "weights_gathered":
        h = ag("mk,kn->mn", "rhs", "k", w1_parts, x_shards)
        return ag("mk,kn->mn", "rhs", "k", w2_parts, h)
    raise ValueError(f"unknown reading {reading!r}")


def mesh_device(x, y, n_y):
    """Device index of mesh coordinate (x, y) on an [M, N] mesh: d = x * N + y."""
    return x * n_y + y


def mlp_2d_reference(x_full, w1_full, w2_full, m_x, n_y):
    """Unpartitioned Y = X @ W1 @ W2, cut into the per-device output blocks.

    Device (x, y) holds Y's y-th row block (batch / N) and x-th column block
    (F / M): the same layout as its input activations.
    """
    y_full = mlp_1d_reference(x_full, w1_full, w2_full)
    rows = np.split(y_full, n_y, axis=0)
    return {(x, y): np.split(rows[y], m_x, axis=1)[x] for x in range(m_x) for y in range(n_y)}


def mlp_2d_forward(x_blocks, w1_blocks, w2_blocks, m_x, n_y, looped=True):
    """Two-layer MLP on an [M, N] mesh ([Decomp] §2.2, Fig. 3).

    The figure's tensor shapes are not printed; the reading used is:
    X(x,y) = [B/N, F/M], W1(x,y) = [F/N, H/M], W2(x,y) = [H/M, F/N], i.e.
    X = blocks (batch by y, feature by x), W1 = blocks (F by y, H by x),
    W2 = blocks (H by x, F by y). Arguments are dicts keyed by (x, y).

    1. AllGather X along x (its feature dimension): [B/N, F].
    2. Looped AllGather-Einsum of W1 along y over its contracting dimension F
       (case 2, looped operand on the right): h(x,y) = [B/N, H/M].
    3. AllGather W2 along y (its F dimension): [H/M, F].
    4. Looped Einsum-ReduceScatter along x (the subgroup ReduceScatter of the
       figure) on the F dimension of the output: y(x,y) = [B/N, F/M].

    The batch dimension stays partitioned throughout, activations and weights
    are gathered along different mesh axes, and the output has X's layout, as
    the section describes. Returns a dict keyed by (x, y).
    """
    ag = looped_allgather_einsum if looped else allgather_einsum
    rs = looped_einsum_reduce_scatter if looped else einsum_reduce_scatter
    xf = {}
    for y in range(n_y):  # step 1, subgroups of fixed y
        full = allgather([x_blocks[(x, y)] for x in range(m_x)], 1)
        for x in range(m_x):
            xf[(x, y)] = full
    h = {}
    for x in range(m_x):  # step 2, subgroups of fixed x
        outs = ag("mk,kn->mn", "rhs", "k",
                  [w1_blocks[(x, y)] for y in range(n_y)],
                  [xf[(x, y)] for y in range(n_y)])
        for y in range(n_y):
            h[(x, y)] = outs[y]
    w2f = {}
    for x in range(m_x):  # step 3, subgroups of fixed x
        full = allgather([w2_blocks[(x, y)] for y in range(n_y)], 1)
        for y in range(n_y):
            w2f[(x, y)] = full
    out = {}
    for y in range(n_y):  # step 4, subgroups of fixed y
        ys = rs("mk,kn->mn",
                [h[(x, y)] for x in range(m_x)],
                [w2f[(x, y)] for x in range(m_x)], "n")
        for x in range(m_x):
            out[(x, y)] = ys[x]
    return out


def megatron_attention_tail(in_slices, w_slices, bias, residual, p, seed):
    """[CoCoNet] Fig. 3: ``layer = MatMul(in, w)`` with ``in`` sliced on its
    last dimension and ``w`` on its first (a local result), then
    ``FusedAllReduce`` with bias, dropout and residual. Returns (layer list,
    replicated output)."""
    layers = [einsum("mk,kn->mn", a, b) for a, b in zip(in_slices, w_slices)]
    return layers, fused_allreduce(layers, bias, residual, p, seed)
