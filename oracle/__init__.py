"""CPU oracle for the fused and decomposed collectives -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct restatement of what the GPU
path computes, in float64 NumPy. Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it. The product path (``collective_fusedallreduce_gb300``) never imports it and
shares no code with it: no kernels, helpers, tables or constants. The only
thing both sides see is the seeded input data, made by
``collective_fusedallreduce_gb300.synth`` (random numbers only, none of the
method's arithmetic) and handed to each side separately.

Sources, cited by title and section throughout:

* [CoCoNet] "Breaking the Computation and Communication Abstraction Barrier in
  Distributed Machine Learning Workloads" (ASPLOS '22): tensor layouts and the
  Fig. 3 self-attention tail (MatMul -> AllReduce -> +bias -> Dropout ->
  +residual), AllReduce Split RS-AG, AllReduce Fuse / FusedAllReduce (§5.2).
* [Decomp] "Overlap Communication with Dependent Computation via Decomposition
  in Large Deep Learning Models" (ASPLOS '23; the page is a set of notes on the
  paper): §2.1 collective definitions, §2.2 the 1-D / 2-D partitioned MLPs of
  Figs. 2 and 3, §4 the decomposition idea (Figs. 4 and 5), §5.1 the Looped
  CollectiveEinsum (Alg. 1, Figs. 6 and 7) and its three AllGather cases,
  §5.5 the cost model that enables it.

Every function states the passage it follows. Where the pages are silent the
docstring says which reading was taken and why.

Pins: each public function is checked in ``tests/test_oracle_pins.py`` against
facts the pages or mathematics fix (brute force, closed forms, identities the
pages state, published hash test vectors). No function here is unpinned.
"""

from .collectives import (
    allgather,
    reduce_scatter,
    allreduce,
    allreduce_split_rs_ag,
    permute_pairs,
    collective_permute,
)
from .einsum import einsum, einsum_bruteforce, parse_spec
from .looped import (
    allgather_einsum,
    looped_allgather_einsum,
    looped_allgather_einsum_bidirectional,
    einsum_reduce_scatter,
    looped_einsum_reduce_scatter,
    looped_einsum_reduce_scatter_unrolled,
    looped_einsum_reduce_scatter_bidirectional,
)
from .fused import (
    splitmix64,
    counter_hash,
    keep_threshold,
    keep_mask,
    dropout_scale,
    fused_allreduce,
)
from .scattered import (
    buckets as scattered_buckets,
    metadata_bytes as scattered_metadata_bytes,
    scattered_allreduce,
    scattered_allreduce_by_buckets,
)
from .costmodel import loop_profitable
from .mlp import (
    mlp_1d_forward,
    mlp_1d_reference,
    mlp_2d_forward,
    mlp_2d_reference,
    megatron_attention_tail,
)

__all__ = [
    "allgather", "reduce_scatter", "allreduce", "allreduce_split_rs_ag",
    "permute_pairs", "collective_permute",
    "einsum", "einsum_bruteforce", "parse_spec",
    "allgather_einsum", "looped_allgather_einsum", "looped_allgather_einsum_bidirectional",
    "einsum_reduce_scatter", "looped_einsum_reduce_scatter", "looped_einsum_reduce_scatter_unrolled",
    "looped_einsum_reduce_scatter_bidirectional",
    "splitmix64", "counter_hash", "keep_threshold", "keep_mask", "dropout_scale",
    "fused_allreduce",
    "mlp_1d_forward", "mlp_1d_reference", "mlp_2d_forward", "mlp_2d_reference",
    "megatron_attention_tail",
    "scattered_buckets", "scattered_metadata_bytes", "scattered_allreduce", "scattered_allreduce_by_buckets",
    "loop_profitable",
]
