"""AllReduce over scattered (non-contiguous) tensors (test infrastructure only).

[CoCoNet], the section on scattered tensors: data-parallel gradients live in
many separate buffers; instead of copying them into one large buffer, one
kernel reduces them all. Each tensor is cut into buckets of at most 2**10
elements; a bucket is described by a 64-bit tensor address and a 32-bit
offset (12 bytes), so a tensor of N elements costs 12 * ceil(N / 2**10) bytes
of metadata, which the page puts at 0.6 % for BERT's 334 M elements.
"""

import math

import numpy as np

BUCKET = 1 << 10
ENTRY_BYTES = 8 + 4  # 64-bit address + 32-bit offset


def buckets(numels):
    """The bucket list of a list of tensor sizes: (tensor index, element offset, length) per bucket."""
    out = []
    for t, n in enumerate(numels):
        for off in range(0, int(n), BUCKET):
            out.append((t, off, min(BUCKET, int(n) - off)))
    return out


def metadata_bytes(numel):
    """12 * ceil(N / 2**10): bucket metadata of one tensor of N elements (one rank's copy)."""
    return ENTRY_BYTES * math.ceil(int(numel) / BUCKET)


def scattered_allreduce(per_rank, alpha=1.0):
    """``per_rank[r][t]`` is rank r's tensor t. Every rank ends with
    ``alpha * sum_r per_rank[r][t]`` for every t (summed in rank order,
    float64). Returns the list of reduced tensors (one per t)."""
    n_t = len(per_rank[0])
    out = []
    for t in range(n_t):
        acc = None
        for r in range(len(per_rank)):
            x = np.asarray(per_rank[r][t], np.float64)
            acc = x.copy() if acc is None else acc + x
        out.append(acc * alpha)
    return out


def scattered_allreduce_by_buckets(per_rank, alpha=1.0):
    """The same reduction walked bucket by bucket over the flattened tensors
    (the order the kernel's warps take); equal to ``scattered_allreduce``."""
    numels = [np.asarray(x).size for x in per_rank[0]]
    flat_out = [np.zeros(n) for n in numels]
    for t, off, ln in buckets(numels):
        acc = None
        for r in range(len(per_rank)):
            x = np.asarray(per_rank[r][t], np.float64).ravel()[off:off + ln]
            acc = x.copy() if acc is None else acc + x
        flat_out[t][off:off + ln] = acc * alpha
    return [f.reshape(np.asarray(x).shape) for f, x in zip(flat_out, per_rank[0])]
