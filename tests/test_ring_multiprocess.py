"""The one-rank-per-process Looped CollectiveEinsum and FusedAllReduce
(``collective_fusedallreduce_gb300.ring``) on CPU: gloo, world sizes 2, 3 and 4.

Each rank is a process that owns only its own shards; every CollectivePermute,
all-to-all and all-gather goes through torch.distributed. The steps'
arithmetic, which the product runs in the library's CUDA kernels, is done here
by a float64 NumPy stand-in defined in this file (the kernels themselves are
covered by the GPU tests, including the same loops on one GPU through the
loopback transport). What is checked is the host logic of the ring: the
permute direction and double buffers, the shard IDs that travel with the data
(against the library's schedule and the oracle's trace), DynamicSlice /
DynamicUpdateSlice offsets, the order of the ReduceScatter's additions, the
FusedAllReduce's slices and element indices, and the §5.5 gate's fallback.
World size 3 tells the permute direction apart ({j -> j-1} and {j -> j+1}
coincide for 2 ranks); world size 4 takes the even-N ends of the bidirectional
and unroll-by-2 schedules.
"""

import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class NumpyCompute:
    """The steps of ring.py on CPU tensors, in float64, rounded to the output's type."""

    @staticmethod
    def _f64(t):
        return t.detach().to(torch.float64).numpy()

    @staticmethod
    def _store(dst, v):
        dst.copy_(torch.from_numpy(np.ascontiguousarray(v)).to(dst.dtype))

    def einsum(self, spec, lhs, rhs, out):
        import oracle
        for a, b, o in zip(lhs, rhs, out):
            self._store(o, oracle.einsum(spec, self._f64(a), self._f64(b)))

    def einsum_accumulate(self, spec, lhs, rhs, acc):
        import oracle
        for a, b, c in zip(lhs, rhs, acc):
            self._store(c, self._f64(c) + oracle.einsum(spec, self._f64(a), self._f64(b)))

    def accumulate(self, acc, part):
        for a, p in zip(acc, part):
            self._store(a, self._f64(a) + self._f64(p))

    def assemble(self, chunks, dim, full):
        self._store(full, np.concatenate([self._f64(c) for c in chunks], axis=dim))

    def fused_slice(self, slices, bias, residual, p, seed, index_base, out):
        import oracle
        shape = tuple(slices[0].shape)
        index = index_base + np.arange(int(np.prod(shape)), dtype=np.uint64).reshape(shape)
        v = oracle.fused_allreduce([self._f64(s) for s in slices], None if bias is None else self._f64(bias),
                                   None if residual is None else self._f64(residual), p, seed, index)
        self._store(out, v)


def _inputs(world):
    from collective_fusedallreduce_gb300 import synth
    f32 = torch.float32
    return {
        # case 1: LHS rows sliced (m), each rank's own RHS
        "c1_shards": synth.per_rank(71, 0, world, (4, 8), f32, "smallint"),
        "c1_rhs": synth.per_rank(71, 1, world, (8, 6), f32, "smallint"),
        # case 2: LHS sliced on the contracting dimension k, RHS DynamicSliced along k
        "c2_shards": synth.per_rank(71, 2, world, (4, 3), f32, "smallint"),
        "c2_rhs": synth.per_rank(71, 3, world, (3 * world, 5), f32, "smallint"),
        # case 3: batched LHS sliced on the batch
        "c3_shards": synth.per_rank(71, 4, world, (2, 3, 4), f32, "smallint"),
        "c3_rhs": synth.per_rank(71, 5, world, (2 * world, 4, 5), f32, "smallint"),
        # Einsum-ReduceScatter onto the LHS rows
        "rs_lhs": synth.per_rank(71, 6, world, (2 * world, 3), f32, "smallint"),
        "rs_rhs": synth.per_rank(71, 7, world, (3, 4), f32, "smallint"),
        # FusedAllReduce
        "far_partials": synth.per_rank(71, 8, world, (2 * world, 16), f32, "uniform"),
        "far_bias": synth.tensor(synth.seed_of(71, 9), (16,), f32, "uniform"),
        "far_res": synth.tensor(synth.seed_of(71, 10), (2 * world, 16), f32, "uniform"),
    }


def _worker(rank, world, port, q):
    try:
        _run(rank, world, port, q)
    except BaseException:  # report instead of leaving the parent waiting
        import traceback
        q.put((rank, {"error": traceback.format_exc()}))
        raise


def _run(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import oracle
    from collective_fusedallreduce_gb300 import ring
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=__import__("datetime").timedelta(seconds=60))
    try:
        T = ring.DistTransport()
        C = NumpyCompute()
        x = _inputs(world)
        f64 = NumpyCompute._f64
        res = {}

        def ag(key, spec, lab, out_shape, gate=None):
            trace = []
            out = [torch.zeros(out_shape)]
            ring.looped_allgather_einsum(spec, "lhs", lab, [x[key + "_shards"][rank]], [x[key + "_rhs"][rank]],
                                         out, T, C, trace=None if gate is not None else trace, gate=gate)
            otrace = []
            want = oracle.looped_allgather_einsum(spec, "lhs", lab, [f64(s) for s in x[key + "_shards"]],
                                                  [f64(r) for r in x[key + "_rhs"]], otrace)[rank]
            mine = sorted(t for t in otrace if t[1] == rank)
            return bool(np.array_equal(f64(out[0]), want)), (gate is not None or sorted(trace) == mine)

        res["case1"] = ag("c1", "mk,kn->mn", "m", (4 * world, 6))
        res["case2"] = ag("c2", "mk,kn->mn", "k", (4, 5))
        res["case3"] = ag("c3", "bmk,bkn->bmn", "b", (2 * world, 3, 5))
        # §5.5 gate: a ring slower than the computation can hide keeps the original AllGather + einsum
        keep = (1.0, 1.0, 5.0, 0.0)
        assert not ring.decompose(keep)
        res["case1_gated"] = ag("c1", "mk,kn->mn", "m", (4 * world, 6), gate=keep)
        res["case3_gated"] = ag("c3", "bmk,bkn->bmn", "b", (2 * world, 3, 5), gate=keep)

        trace = []
        out = [torch.zeros((2, 4))]
        ring.looped_einsum_reduce_scatter("mk,kn->mn", [x["rs_lhs"][rank]], [x["rs_rhs"][rank]], out, T, C, trace)
        otrace = []
        want = oracle.looped_einsum_reduce_scatter("mk,kn->mn", [f64(a) for a in x["rs_lhs"]],
                                                   [f64(b) for b in x["rs_rhs"]], "m", otrace)[rank]
        res["rs"] = (bool(np.array_equal(f64(out[0]), want)), sorted(trace) == sorted(t for t in otrace if t[1] == rank))
        kept = [torch.zeros((2, 4))]
        ring.looped_einsum_reduce_scatter("mk,kn->mn", [x["rs_lhs"][rank]], [x["rs_rhs"][rank]], kept, T, C, gate=keep)
        res["rs_gated"] = (bool(np.array_equal(f64(kept[0]), want)), True)

        # the section 5.4 schedules: bidirectional AllGather-Einsum (cases 1, 2, 3), unroll-by-2 and
        # bidirectional Einsum-ReduceScatter, each against the oracle's restatement and its shard IDs
        for key, spec, lab, shape in (("c1", "mk,kn->mn", "m", (4 * world, 6)), ("c2", "mk,kn->mn", "k", (4, 5)),
                                      ("c3", "bmk,bkn->bmn", "b", (2 * world, 3, 5))):
            trace, otrace = [], []
            out = [torch.zeros(shape)]
            ring.looped_allgather_einsum(spec, "lhs", lab, [x[key + "_shards"][rank]], [x[key + "_rhs"][rank]], out,
                                         T, C, trace=trace, schedule=2)
            want = oracle.looped_allgather_einsum_bidirectional(spec, "lhs", lab, [f64(v) for v in x[key + "_shards"]],
                                                                [f64(v) for v in x[key + "_rhs"]], otrace)[rank]
            res[key + "_bidirectional"] = (bool(np.array_equal(f64(out[0]), want)),
                                           sorted(trace) == sorted(t for t in otrace if t[1] == rank))
        for sched, fn in ((1, oracle.looped_einsum_reduce_scatter_unrolled),
                          (2, oracle.looped_einsum_reduce_scatter_bidirectional)):
            trace, otrace = [], []
            out = [torch.zeros((2, 4))]
            ring.looped_einsum_reduce_scatter("mk,kn->mn", [x["rs_lhs"][rank]], [x["rs_rhs"][rank]], out, T, C,
                                              trace, schedule=sched)
            want = fn("mk,kn->mn", [f64(v) for v in x["rs_lhs"]], [f64(v) for v in x["rs_rhs"]], "m", otrace)[rank]
            res[f"rs_sched{sched}"] = (bool(np.array_equal(f64(out[0]), want)),
                                       sorted(trace) == sorted(t for t in otrace if t[1] == rank))

        out = [torch.empty((2 * world, 16))]
        ring.fused_allreduce([x["far_partials"][rank]], x["far_bias"], [x["far_res"]], 0.25, 1234, out, T, C)
        want = oracle.fused_allreduce([f64(p) for p in x["far_partials"]], f64(x["far_bias"]), f64(x["far_res"]),
                                      0.25, 1234).astype(np.float32)
        dropped = ~oracle.keep_mask(1234, 0.25, np.arange(want.size, dtype=np.uint64)).reshape(want.shape)
        res["far"] = (bool(np.array_equal(out[0].numpy(), want)),
                      bool(np.array_equal(out[0].numpy()[dropped], x["far_res"].numpy()[dropped])))
        q.put((rank, res))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("world", [2, 3, 4])
def test_ring_over_gloo_matches_the_oracle(world):
    import __graft_entry__
    __graft_entry__.build()  # the schedule comes from the library (host-only calls)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(120)
    for rank in range(world):
        assert "error" not in got[rank], got[rank]["error"]
    for p in procs:
        assert p.exitcode == 0
    for rank in range(world):
        for name, (equal, sched) in got[rank].items():
            assert equal, (rank, name, "result differs from the oracle")
            assert sched, (rank, name, "shard IDs differ from the oracle's schedule")


def test_cost_model_times_and_decision():
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import ring
    # 1 TFLOP einsum at 1000 TFLOP/s = 1 ms; 7 shards of 100 MB: 0.7 GB over 700 GB/s (collective) = 1 ms,
    # over one 350 GB/s link = 2 ms
    comp, comm, ring_t, epi = ring.ring_times(1e12, 100e6, 8, 1000.0, 350.0, 700.0)
    assert abs(comp - 1e-3) < 1e-12 and abs(comm - 1e-3) < 1e-12 and abs(ring_t - 2e-3) < 1e-12 and epi == 0.0
    assert ring.decompose((comp, comm, ring_t, epi))            # 2 ms >= max(1, 2) ms
    assert not ring.decompose((comp, comm, ring_t, 1e-6))      # any epilogue tips it
    assert ring.decompose(ring.ring_times(4e12, 100e6, 8, 1000.0, 350.0, 700.0, 1e-3))


def test_compute_on_cpu_tensors_fails_loudly():
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    from collective_fusedallreduce_gb300 import ring
    with pytest.raises(RuntimeError, match="GPU"):
        ring.CocoCompute().einsum("mk,kn->mn", [torch.zeros(8, 8)], [torch.zeros(8, 8)], [torch.zeros(8, 8)])
