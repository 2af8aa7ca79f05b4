"""The enabling rule of the Looped CollectiveEinsum (test infrastructure only).

[Decomp] "Overlap Communication with Dependent Computation via Decomposition
in Large Deep Learning Models", §5.5 (cost model and enabling mechanism): the
decomposed loop moves its shards along one logical ring, which can use less
of the interconnect than the original collective on a mesh or torus, so it
is applied only where the estimate says it pays. The rule compares the
original einsum and collective, run one after the other, with the loop, in
which the einsum and the ring transfers overlap and a prologue or epilogue is
added.
"""


def loop_profitable(orig_comp, orig_comm, ring_comm, epilogue_cost):
    """True when the original computation time plus the original communication
    time is at least the larger of the computation time and the ring's
    communication time, plus the prologue / epilogue cost (the §5.5
    inequality, taken with "at least" as printed). Times are non-negative
    numbers in one unit."""
    for t in (orig_comp, orig_comm, ring_comm, epilogue_cost):
        if not (t >= 0.0) or t == float("inf"):
            raise ValueError("times must be finite and non-negative")
    original = orig_comp + orig_comm
    looped = max(orig_comp, ring_comm) + epilogue_cost
    return original >= looped
