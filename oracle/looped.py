"""AllGather-Einsum and Einsum-ReduceScatter, monolithic and looped (test infrastructure only).

Monolithic forms follow the unfused semantics: the full collective, then the
einsum ([Decomp] §2.2, Fig. 2). Looped forms restate the Looped
CollectiveEinsum of [Decomp] §4 (Figs. 4 and 5) and §5.1 (Alg. 1, Figs. 6 and
7) with explicit permute buffers: N iterations, each a partial einsum on the
shard whose ID travels with the data, an Update (DynamicUpdateSlice or
Addition), and a CollectivePermute along the pairs {j -> j-1 mod N}.

The page prints Alg. 1's caption but not its body. The body is reconstructed
from the prose of §4 and §5.1, read as follows:

* AllGather: rank r starts with its own shard (shard IDs aligned with
  partition IDs at the loop start), computes, updates, and passes the shard to
  rank r-1 after every iteration but the last.
* ReduceScatter: every rank starts with a zero accumulator tagged with its own
  partition ID. At the start of each iteration it sends the accumulator to
  rank r-1; it then computes the partial einsum for the shard ID of the
  accumulator it receives and adds it. After N iterations each rank holds the
  accumulator of its own partition ID (aligned at the loop end), and the
  DynamicSlice index a rank uses first is not its own partition ID.

An optional ``trace`` list receives ``(iteration, rank, shard_id)`` tuples so
tests can check the schedule against the pages' description.
"""

import numpy as np

from .collectives import allgather, reduce_scatter, permute_pairs, collective_permute
from .einsum import einsum, parse_spec


def _slice(arr, dim, index, size):
    """DynamicSlice: ``size`` entries of ``arr`` along ``dim`` starting at ``index * size``."""
    sl = [slice(None)] * arr.ndim
    sl[dim] = slice(index * size, (index + 1) * size)
    return arr[tuple(sl)]


def _apply(spec, looped, looped_val, other_val):
    return einsum(spec, looped_val, other_val) if looped == "lhs" else einsum(spec, other_val, looped_val)


def allgather_einsum(spec, looped, slice_label, shards, locals_):
    """Monolithic AllGather -> Einsum: gather the sliced operand, then contract.

    ``looped`` is ``"lhs"`` or ``"rhs"``: which operand is sliced over the
    ranks. ``slice_label`` is the spec letter of its sliced dimension.
    ``shards[s]`` is shard s of that operand; ``locals_[r]`` is rank r's other
    operand (distinct per rank for a local tensor, equal for a replicated
    one). Returns ``[out_r]``.
    """
    lab_l, lab_r, _ = parse_spec(spec)
    labels = lab_l if looped == "lhs" else lab_r
    full = allgather(shards, labels.index(slice_label))
    return [_apply(spec, looped, full, np.asarray(loc, np.float64)) for loc in locals_]


def looped_allgather_einsum(spec, looped, slice_label, shards, locals_, trace=None):
    """Looped AllGather-Einsum ([Decomp] §5.1, the three AllGather cases).

    With the looped operand sliced along ``slice_label``:

    * a non-contracting dimension (m of the LHS, n of the RHS) is case 1: the
      partial einsum uses the received shard and the whole other operand, and a
      DynamicUpdateSlice writes the shard's rows (columns) of the result;
    * the contracting dimension k is case 2: the other operand is DynamicSliced
      along k with the shard's size, and the Update is an Addition;
    * the batch dimension b is case 3: the other operand is DynamicSliced along
      b and a DynamicUpdateSlice along b writes the result.
    """
    n = len(shards)
    lab_l, lab_r, lab_o = parse_spec(spec)
    looped_labels = lab_l if looped == "lhs" else lab_r
    other_labels = lab_r if looped == "lhs" else lab_l
    if slice_label not in looped_labels:
        raise ValueError(f"{slice_label!r} is not a dimension of the {looped} operand")
    shard_extent = np.asarray(shards[0]).shape[looped_labels.index(slice_label)]
    update = "add" if slice_label == "k" else "dus"

    held = [(r, np.asarray(shards[r], np.float64)) for r in range(n)]
    outs = [None] * n
    for i in range(n):
        for r in range(n):
            sid, data = held[r]
            other = np.asarray(locals_[r], np.float64)
            if slice_label in other_labels:  # cases 2 and 3: DynamicSlice the other operand
                other = _slice(other, other_labels.index(slice_label), sid, shard_extent)
            partial = _apply(spec, looped, data, other)
            if trace is not None:
                trace.append((i, r, sid))
            if update == "add":
                outs[r] = partial.copy() if outs[r] is None else outs[r] + partial
            else:
                o = lab_o.index(slice_label)
                if outs[r] is None:
                    shape = list(partial.shape)
                    shape[o] *= n
                    outs[r] = np.zeros(shape)
                sl = [slice(None)] * partial.ndim
                sl[o] = slice(sid * shard_extent, (sid + 1) * shard_extent)
                outs[r][tuple(sl)] = partial
        if i < n - 1:
            held = collective_permute(held, permute_pairs(n))
    return outs


def einsum_reduce_scatter(spec, lhs_list, rhs_list, out_label):
    """Monolithic Einsum -> ReduceScatter: every rank contracts its own
    operands (both sliced on the contracting dimension, so the result is a
    local partial sum, [CoCoNet] layout rule for MatMul), then the partials
    are reduce-scattered along the output dimension ``out_label``.
    """
    _, _, lab_o = parse_spec(spec)
    partials = [einsum(spec, l, r) for l, r in zip(lhs_list, rhs_list)]
    return reduce_scatter(partials, lab_o.index(out_label))


def _rs_sliced_operand(spec, out_label):
    """[Decomp] §5.1 Einsum-ReduceScatter rule: the operand that owns the
    non-contracting dimension the output is partitioned on is the one that is
    DynamicSliced."""
    lab_l, lab_r, _ = parse_spec(spec)
    if out_label == "k" or out_label == "b":
        raise ValueError("the output must be partitioned on a non-contracting, non-batch dimension")
    if out_label in lab_l:
        return "lhs", lab_l.index(out_label)
    return "rhs", lab_r.index(out_label)


def looped_einsum_reduce_scatter(spec, lhs_list, rhs_list, out_label, trace=None):
    """Looped Einsum-ReduceScatter ([Decomp] §4 Fig. 5 and §5.1).

    The transferred data is the accumulated result shard. Each rank starts
    with a zero accumulator; at the start of every iteration it sends it to
    rank r-1, computes the partial einsum for the shard ID of the accumulator
    it receives (DynamicSlice of the operand that owns ``out_label``), and
    adds it. Returns ``[y_r]``; raises if the final shard IDs are not aligned
    with the partition IDs.
    """
    n = len(lhs_list)
    _, _, lab_o = parse_spec(spec)
    side, dim = _rs_sliced_operand(spec, out_label)
    lhs_list = [np.asarray(x, np.float64) for x in lhs_list]
    rhs_list = [np.asarray(x, np.float64) for x in rhs_list]
    full_extent = (lhs_list if side == "lhs" else rhs_list)[0].shape[dim]
    if full_extent % n:
        raise ValueError("output dimension does not split into equal shards")
    size = full_extent // n

    probe = einsum(spec, lhs_list[0], rhs_list[0])
    shard_shape = list(probe.shape)
    shard_shape[lab_o.index(out_label)] = size
    acc = [(r, np.zeros(shard_shape)) for r in range(n)]
    for i in range(n):
        acc = collective_permute(acc, permute_pairs(n))
        for q in range(n):
            sid, a = acc[q]
            if side == "lhs":
                partial = einsum(spec, _slice(lhs_list[q], dim, sid, size), rhs_list[q])
            else:
                partial = einsum(spec, lhs_list[q], _slice(rhs_list[q], dim, sid, size))
            if trace is not None:
                trace.append((i, q, sid))
            acc[q] = (sid, a + partial)
    for r, (sid, _) in enumerate(acc):
        if sid != r:
            raise AssertionError(f"rank {r} ends with shard {sid}: not aligned at the loop end")
    return [a for _, a in acc]


# ------------------------------------------------------------------------------
# Schedule variants of [Decomp] §5.4: loop unrolling by 2 (§5.4.1, Fig. 8) and
# bidirectional data transfer (§5.4.2, Figs. 9 and 10). Both are presented as
# optimisations that keep the loop semantically equivalent; the figures are not
# printed, so the schedules below are restated from the prose (a reading of it).
# Shard IDs travel with the data as in the ring forms above.


def _update(out, partial, update, o, sid, extent, n):
    if update == "add":
        return partial.copy() if out is None else out + partial
    if out is None:
        shape = list(partial.shape)
        shape[o] *= n
        out = np.zeros(shape)
    sl = [slice(None)] * partial.ndim
    sl[o] = slice(sid * extent, (sid + 1) * extent)
    out[tuple(sl)] = partial
    return out


def bidirectional_pairs(n, direction):
    """Permute pairs moving data left ({j -> j-1}) or right ({j -> j+1})."""
    return [(src, (src - 1) % n) if direction == "left" else (src, (src + 1) % n) for src in range(n)]


def looped_allgather_einsum_bidirectional(spec, looped, slice_label, shards, locals_, trace=None):
    """Bidirectional Looped AllGather-Einsum ([Decomp] §5.4.2, Fig. 9).

    Prologue: every rank computes with its own shard and sends it both ways.
    Then each iteration k = 1, 2, ... receives one shard from each direction
    (shards r+k and r-k), computes with both in one step (the concatenated
    einsum of the page), and forwards each in its own direction. With N even
    the last shard (r + N/2) arrives from one side only and is used once.
    ``trace`` gets (step, rank, shard_id) for every shard used.
    """
    n = len(shards)
    lab_l, lab_r, lab_o = parse_spec(spec)
    looped_labels = lab_l if looped == "lhs" else lab_r
    other_labels = lab_r if looped == "lhs" else lab_l
    extent = np.asarray(shards[0]).shape[looped_labels.index(slice_label)]
    update = "add" if slice_label == "k" else "dus"
    o = lab_o.index(slice_label) if update == "dus" else None

    def partial_for(r, sid, data):
        other = np.asarray(locals_[r], np.float64)
        if slice_label in other_labels:
            other = _slice(other, other_labels.index(slice_label), sid, extent)
        return _apply(spec, looped, data, other)

    outs = [None] * n
    own = [(r, np.asarray(shards[r], np.float64)) for r in range(n)]
    for r in range(n):  # prologue: the own shard
        sid, data = own[r]
        outs[r] = _update(outs[r], partial_for(r, sid, data), update, o, sid, extent, n)
        if trace is not None:
            trace.append((0, r, sid))
    left, right = own, own
    step = 1
    used = 1
    while used < n:
        left = collective_permute(left, bidirectional_pairs(n, "left"))    # from r+1: shard r+step
        right = collective_permute(right, bidirectional_pairs(n, "right"))  # from r-1: shard r-step
        for r in range(n):
            got = [left[r]]
            if used + 1 < n:
                got.append(right[r])
            partial = None
            for sid, data in got:  # the two halves of one concatenated step
                p = partial_for(r, sid, data)
                if update == "add":
                    partial = p if partial is None else partial + p
                else:
                    outs[r] = _update(outs[r], p, update, o, sid, extent, n)
                if trace is not None:
                    trace.append((step, r, sid))
            if update == "add":
                outs[r] = outs[r] + partial
        used += 2 if used + 1 < n else 1
        step += 1
    return outs


def _rs_partial_fn(spec, lhs_list, rhs_list, out_label):
    n = len(lhs_list)
    side, dim = _rs_sliced_operand(spec, out_label)
    lhs_list = [np.asarray(x, np.float64) for x in lhs_list]
    rhs_list = [np.asarray(x, np.float64) for x in rhs_list]
    size = (lhs_list if side == "lhs" else rhs_list)[0].shape[dim] // n

    def partial(q, sid):
        if side == "lhs":
            return einsum(spec, _slice(lhs_list[q], dim, sid, size), rhs_list[q])
        return einsum(spec, lhs_list[q], _slice(rhs_list[q], dim, sid, size))

    return partial


def _check_aligned(chain):
    for r, (sid, _) in enumerate(chain):
        if sid != r:
            raise AssertionError(f"rank {r} holds shard {sid} after the epilogue")


def looped_einsum_reduce_scatter_unrolled(spec, lhs_list, rhs_list, out_label, trace=None):
    """Looped Einsum-ReduceScatter unrolled by 2 ([Decomp] §5.4.1, Fig. 8).

    The accumulation chain is split into two interleaved chains that travel
    the ring two hops per iteration ({j -> j-2}): chain A collects ranks
    r-1, r-3, ... and chain B ranks r-2, r-4, ... of output shard r (together
    every rank once). An epilogue moves the chain that ends one hop short
    onto rank r and adds the two chains there.
    ``trace`` gets (iteration, rank, chain, shard_id).
    """
    n = len(lhs_list)
    partial = _rs_partial_fn(spec, lhs_list, rhs_list, out_label)
    shape = list(partial(0, 0).shape)
    two_hops = [(src, (src - 2) % n) for src in range(n)]
    chain_a = [((q + 1) % n, np.zeros(shape)) for q in range(n)]  # rank q first adds to shard q+1
    chain_b = [((q + 2) % n, np.zeros(shape)) for q in range(n)]  # and to shard q+2
    n_a, n_b = (n + 1) // 2, n // 2
    for i in range(n_a):
        if i > 0:
            chain_a = collective_permute(chain_a, two_hops)
            if i < n_b:
                chain_b = collective_permute(chain_b, two_hops)
        for q in range(n):
            sid, acc = chain_a[q]
            chain_a[q] = (sid, acc + partial(q, sid))
            if trace is not None:
                trace.append((i, q, "A", sid))
            if i < n_b:
                sid, acc = chain_b[q]
                chain_b[q] = (sid, acc + partial(q, sid))
                if trace is not None:
                    trace.append((i, q, "B", sid))
    # epilogue: the chain whose last contribution came from rank r+1 takes one more hop
    one_hop = permute_pairs(n)
    if n % 2 == 0:
        chain_a = collective_permute(chain_a, one_hop)
    elif n > 1:
        chain_b = collective_permute(chain_b, one_hop)
    _check_aligned(chain_a)
    if n > 1:
        _check_aligned(chain_b)
        return [a + b for (_, a), (_, b) in zip(chain_a, chain_b)]
    return [a for _, a in chain_a]


def looped_einsum_reduce_scatter_bidirectional(spec, lhs_list, rhs_list, out_label, trace=None):
    """Bidirectional Looped Einsum-ReduceScatter ([Decomp] §5.4.2, Fig. 10).

    Output shard r has two accumulators travelling in opposite directions: a
    left-moving one ({j -> j-1}) that collects ranks r+a, r+a-1, ..., r+1 and
    a right-moving one ({j -> j+1}) that collects ranks r-b, ..., r-1, with
    a = ceil((N-1)/2) and b = floor((N-1)/2). The epilogue moves each one hop
    onto rank r, which adds both to its own partial.
    ``trace`` gets (iteration, rank, direction, shard_id).
    """
    n = len(lhs_list)
    partial = _rs_partial_fn(spec, lhs_list, rhs_list, out_label)
    shape = list(partial(0, 0).shape)
    a, b = n // 2, (n - 1) // 2
    left = [((q - a) % n, np.zeros(shape)) for q in range(n)]   # rank q first adds to shard q-a
    right = [((q + b) % n, np.zeros(shape)) for q in range(n)]  # and to shard q+b
    for i in range(max(a, b)):
        if i > 0:
            if i < a:
                left = collective_permute(left, bidirectional_pairs(n, "left"))
            if i < b:
                right = collective_permute(right, bidirectional_pairs(n, "right"))
        for q in range(n):
            if i < a:
                sid, acc = left[q]
                left[q] = (sid, acc + partial(q, sid))
                if trace is not None:
                    trace.append((i, q, "left", sid))
            if i < b:
                sid, acc = right[q]
                right[q] = (sid, acc + partial(q, sid))
                if trace is not None:
                    trace.append((i, q, "right", sid))
    outs = [partial(r, r) for r in range(n)]  # each rank's own contribution
    if a:
        left = collective_permute(left, bidirectional_pairs(n, "left"))
        _check_aligned(left)
        outs = [o + acc for o, (_, acc) in zip(outs, left)]
    if b:
        right = collective_permute(right, bidirectional_pairs(n, "right"))
        _check_aligned(right)
        outs = [o + acc for o, (_, acc) in zip(outs, right)]
    return outs
