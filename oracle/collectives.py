"""Collective definitions over N logical ranks, in float64 (test infrastructure only).

A "rank's buffer" is one NumPy array; a collective takes a list of them indexed
by rank (partition ID). Definitions follow [Decomp] §2.1 ("Communication
primitives") and [CoCoNet]'s AllReduce Split RS-AG transformation.
"""

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def allgather(shards, dim):
    """AllGather ([Decomp] §2.1): every partition receives the data of all
    partitions, concatenated in partition-ID order along ``dim``.

    ``shards[r]`` is rank r's slice. Returns the gathered array (the same on
    every rank: a replicated tensor in [CoCoNet]'s layout terms).
    """
    return np.concatenate([_f64(s) for s in shards], axis=dim)


def reduce_scatter(locals_, dim):
    """ReduceScatter ([Decomp] §2.1): the inverse communication pattern of
    AllGather. Every rank cuts its local tensor into N equal shards along
    ``dim``; rank r receives shard r from every rank and reduces them element
    by element (sum). Returns ``[out_0, ..., out_{N-1}]``.

    The received shards are summed in rank order q = 0, 1, ..., N-1.
    Uneven division is rejected: [CoCoNet] defines a sliced tensor as
    "equally distributed" over the ranks.
    """
    n = len(locals_)
    extent = _f64(locals_[0]).shape[dim]
    if extent % n:
        raise ValueError(f"dimension {dim} of size {extent} does not split into {n} equal shards")
    outs = []
    for r in range(n):
        acc = None
        for q in range(n):
            shard = np.split(_f64(locals_[q]), n, axis=dim)[r]
            acc = shard.copy() if acc is None else acc + shard
        outs.append(acc)
    return outs


def allreduce(locals_):
    """AllReduce ([Decomp] §2.1; [CoCoNet] Fig. 3 line 9): the element-wise
    sum over all ranks, returned on every rank (replicated layout).

    Summation order: rank 0, 1, ..., N-1. Returns a list of N equal arrays.
    """
    acc = None
    for x in locals_:
        acc = _f64(x).copy() if acc is None else acc + _f64(x)
    return [acc.copy() for _ in locals_]


def allreduce_split_rs_ag(locals_, dim=0):
    """AllReduce Split RS-AG ([CoCoNet], split transformation): a
    ReduceScatter producing a sliced tensor, followed by an AllGather of that
    sliced tensor producing a replicated one. [Decomp] §2.1 states the same
    identity (AllReduce = ReduceScatter then AllGather).
    """
    shards = reduce_scatter(locals_, dim)
    full = allgather(shards, dim)
    return [full.copy() for _ in locals_]


def permute_pairs(n):
    """The {source, destination} pairs of one CollectivePermute step of the
    Looped CollectiveEinsum ([Decomp] §5.1): {0, N-1}, {1, 0}, {2, 1}, ...,
    {N-1, N-2}. Data moves one position to the left around the ring.
    """
    return [(src, (src - 1) % n) for src in range(n)]


def collective_permute(buffers, pairs):
    """CollectivePermute ([Decomp] §2.1): point-to-point transfer between each
    listed (source, destination) pair. ``buffers[r]`` is whatever rank r sends
    (any Python object; the looped algorithms send (shard_id, array) pairs so
    the ID travels with the data). A rank that is no pair's destination keeps
    ``None``.
    """
    out = [None] * len(buffers)
    for src, dst in pairs:
        out[dst] = buffers[src]
    return out
