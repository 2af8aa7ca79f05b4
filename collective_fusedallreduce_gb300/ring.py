"""The Looped CollectiveEinsum and the FusedAllReduce with one rank per device.

In the rest of this package all N logical ranks live in one GPU's memory and a
CollectivePermute is a read of the shard where it lives. Here every rank
owns its buffers and the data really moves:

* [Decomp] "Overlap Communication with Dependent Computation via
  Decomposition in Large Deep Learning Models", §4 (Figs. 4 and 5) and §5.1
  (Alg. 1): N iterations, each starting an asynchronous CollectivePermute
  along the pairs {j -> j-1} into a local receive buffer (the double buffer
  of §5.4.1), computing the partial einsum of the shard in hand while the
  transfer runs, then waiting for it (CollectivePermuteDone). AllGather-
  Einsum: cases 1, 2 and 3 of §5.1; Einsum-ReduceScatter: the accumulator
  travels and each rank adds its partial for the shard ID it receives.
* [Decomp] §5.4: the bidirectional AllGather-Einsum and the unroll-by-2 and
  bidirectional Einsum-ReduceScatter, with their chains travelling in both
  directions or two hops at a time.
* [Decomp] §5.5: the loop replaces the original collective + einsum only when
  the cost model says it pays (coco_loop_profitable); otherwise the original
  operations run (AllGather then one einsum, or the einsum then a
  ReduceScatter).
* [CoCoNet] "Breaking the Computation and Communication Abstraction Barrier
  in Distributed Machine Learning Workloads", AllReduce Split and AllReduce
  Fuse (§5.2): the FusedAllReduce as a ReduceScatter (every rank receives
  slice r of every partial), the bias / dropout / residual on that slice
  only, and an AllGather of the finished slices.

The shard schedule is the library's (coco_shard_order), the one its
single-GPU kernels follow, and the arithmetic of every step runs in the
library's kernels through ``CocoCompute``; the transport only moves bytes.

Transports:
* ``DistTransport``: one rank per process over ``torch.distributed`` (NCCL
  between GPUs, gloo between CPU processes). Point-to-point sends and
  receives, all-to-all and all-gather; no multicast or NVLS.
* ``LoopbackTransport``: all ranks in one process (their buffers in one
  device's memory); a permute is a device copy. It runs the same loops as the
  distributed form, so their schedule and arithmetic can be checked on one
  GPU.

Readings taken where the pages leave a step open:
* The ReduceScatter's first iteration sends a zero accumulator; it carries no
  data, so here iteration 0 writes its partial straight into the accumulator
  and the first transfer happens at iteration 1 (same shard IDs, same sums).
* The distributed Einsum-ReduceScatter accumulates in fp32 (the Addition of
  §5.1 in the accumulator's type) and supports outputs partitioned on the
  rows of the LHS; the FusedAllReduce sums the N slices in rank order 0..N-1
  in fp32, exactly as coco_fused_allreduce does, so the two are bit for bit
  equal.
"""

import torch

from . import coco

AG, RS = coco.AG_ORDER, coco.RS_ORDER


# ------------------------------------------------------------------ transports


class _Done:
    """A started transfer; wait() is the CollectivePermuteDone."""

    def __init__(self, works=()):
        self._works = list(works)

    def wait(self):
        for w in self._works:
            w.wait()
        self._works = []


class DistTransport:
    """One rank per process over torch.distributed (the default process group or ``group``)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self._dist = dist
        self.group = group
        self.nranks = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.local_ranks = [self.rank]

    def _global(self, r):
        return r if self.group is None else self._dist.get_global_rank(self.group, r)

    def permute(self, send, recv, shift=1):
        """Start a CollectivePermute: rank j's ``send`` lands in rank j-shift's ``recv``
        ({j -> j-1} for shift 1). Returns a handle whose wait() completes it."""
        if self.nranks == 1:
            recv[0].copy_(send[0])
            return _Done()
        d = self._dist
        ops = [d.P2POp(d.isend, send[0], self._global((self.rank - shift) % self.nranks), self.group),
               d.P2POp(d.irecv, recv[0], self._global((self.rank + shift) % self.nranks), self.group)]
        return _Done(d.batch_isend_irecv(ops))

    def all_to_all(self, send, recv):
        """Chunk s of recv[0] = chunk r of rank s's send[0] (r = this rank): both are flat tensors of N
        equal chunks."""
        if self.nranks == 1:
            recv[0].copy_(send[0])
            return
        self._dist.all_to_all_single(recv[0], send[0], group=self.group)

    def all_gather(self, src, dst):
        """dst[0][s] = rank s's src."""
        if self.nranks == 1:
            dst[0][0].copy_(src[0])
            return
        self._dist.all_gather(list(dst[0]), src[0], group=self.group)


class LoopbackTransport:
    """All ranks in this process: the per-rank lists hold every rank's tensor."""

    def __init__(self, nranks):
        self.nranks = int(nranks)
        self.rank = None
        self.local_ranks = list(range(self.nranks))

    def permute(self, send, recv, shift=1):
        n = self.nranks
        for j in range(n):
            recv[(j - shift) % n].copy_(send[j])
        return _Done()

    def all_to_all(self, send, recv):
        n = self.nranks
        c = send[0].numel() // n
        for r in range(n):
            for s in range(n):
                recv[r].narrow(0, s * c, c).copy_(send[s].narrow(0, r * c, c))

    def all_gather(self, src, dst):
        for r in range(self.nranks):
            for s in range(self.nranks):
                dst[r][s].copy_(src[s])


# ----------------------------------------------------------------- compute


class CocoCompute:
    """The steps' arithmetic through the library's kernels (CUDA tensors only).

    ``stream``: the CUDA stream the kernels are enqueued on; by default the current stream at each call.
    torch.distributed orders its transfers against the current stream (a transfer starts after the work
    enqueued there, and wait() makes the current stream wait for it), so a different stream is joined to
    the current one around every call: it waits for the current stream's work first, and the current
    stream waits for its kernels afterwards."""

    def __init__(self, stream=None):
        self.stream = stream

    @staticmethod
    def _cuda(ts):
        for t in ts:
            if not t.is_cuda:
                raise RuntimeError("CocoCompute runs the library's CUDA kernels: tensors must be on a GPU")

    def _launch(self, fn, *args):
        s = self.stream
        cur = None if s is None else torch.cuda.current_stream(s.device)
        joined = cur is not None and cur != s
        if joined:
            s.wait_stream(cur)
        fn(*args, s)
        if joined:
            cur.wait_stream(s)

    def einsum(self, spec, lhs, rhs, out):
        """out[l] = lhs[l] @ rhs[l] for every local rank l (one launch)."""
        self._cuda(lhs + rhs + out)
        self._launch(coco.coco_einsum, spec, coco.local(lhs), coco.local(rhs), coco.local(out))

    def einsum_accumulate(self, spec, lhs, rhs, acc):
        """acc[l] += lhs[l] @ rhs[l] (fp32), the Addition done in the einsum's epilogue (one launch)."""
        self._cuda(lhs + rhs + acc)
        self._launch(coco.coco_einsum_accumulate, spec, coco.local(lhs), coco.local(rhs), coco.local(acc))

    def accumulate(self, acc, part):
        """acc[l] = acc[l] + part[l] in the accumulator's type (one launch: a two-rank sum per local rank)."""
        self._cuda(acc + part)
        n = len(acc)
        ins = [t for pair in zip(acc, part) for t in pair]
        outs = [t for a in acc for t in (a, a)]
        self._launch(coco.coco_allreduce, coco.local(ins, ngroups=n), coco.replicated(outs, ngroups=n))

    def assemble(self, chunks, dim, full):
        """full = the chunks concatenated along ``dim`` in partition order (the AllGather's placement)."""
        self._cuda(list(chunks) + [full])
        n = len(chunks)
        self._launch(coco.coco_allgather, coco.sliced(list(chunks), dim), coco.replicated([full] * n))

    def fused_slice(self, slices, bias, residual, p, seed, index_base, out):
        """out = dropout(sum over s of slices[s] + bias) + residual on one slice of the flattened tensor,
        whose first element has whole-tensor index ``index_base``."""
        self._cuda(list(slices) + [out] + ([residual] if residual is not None else []))
        n = len(slices)
        self._launch(coco.coco_fused_allreduce_at, coco.local(list(slices)), bias,
                     None if residual is None else coco.replicated([residual] * n),
                     p, seed, index_base, coco.replicated([out] * n))


# ---------------------------------------------------------- the cost model


def ring_times(flops, shard_bytes, nranks, tensor_tflops, ring_gbs, collective_gbs, epilogue_s=0.0):
    """The four times of [Decomp] §5.5 from a plain bandwidth model: the einsum at the tensor rate, the
    original collective moving (N-1) shards at ``collective_gbs`` (all links of the mesh), the ring moving
    the same (N-1) shards over one link at ``ring_gbs``, and the prologue / epilogue cost given."""
    comp = flops / (tensor_tflops * 1e12)
    moved = (nranks - 1) * shard_bytes
    return comp, moved / (collective_gbs * 1e9), moved / (ring_gbs * 1e9), epilogue_s


def decompose(times):
    """[Decomp] §5.5: decompose only if orig_comp + orig_comm >= max(orig_comp, ring_comm) + epilogue."""
    return coco.coco_loop_profitable(*times)


# ------------------------------------------------- Looped AllGather-Einsum


def _dim(spec, operand, label):
    lhs, rhs = spec.replace(" ", "").split("->")[0].split(",")
    labels = lhs if operand == "lhs" else rhs
    return labels.index(label)


class _Chain:
    """Data travelling around the ring in one direction: the tensors in hand on every local rank, the
    buffers the next transfer lands in (two of the chain's own, so a caller's tensor is only read), and,
    in trace mode, an ID carried beside the data. ``shift`` 1 moves data {j -> j-1}, -1 {j -> j+1},
    2 two hops {j -> j-2}."""

    def __init__(self, first, shift, transport, first_ids=None):
        self.t = transport
        self.shift = shift
        self.cur = list(first)
        self.spare = [[torch.empty_like(x) for x in first] for _ in range(2)]
        self.nxt = self.spare[0]
        self.k = 0
        self.ids = None
        if first_ids is not None:
            dev = first[0].device
            self.ids = [torch.full((1,), int(v), dtype=torch.int64, device=dev) for v in first_ids]
            self.nid = [torch.empty_like(x) for x in self.ids]

    def start(self):  # CollectivePermuteStart
        h = self.t.permute(self.cur, self.nxt, self.shift)
        hid = self.t.permute(self.ids, self.nid, self.shift) if self.ids is not None else None
        return h, hid

    def done(self, hs):  # CollectivePermuteDone: the received data is now in hand
        h, hid = hs
        h.wait()
        self.k += 1
        self.cur, self.nxt = self.nxt, self.spare[self.k % 2]
        if hid is not None:
            hid.wait()
            self.ids, self.nid = self.nid, self.ids

    def check(self, want, what):
        if self.ids is not None:
            got = [int(x.item()) for x in self.ids]
            if got != list(want):
                raise AssertionError(f"{what}: IDs {got} in hand, schedule says {list(want)}")


def looped_allgather_einsum(spec, looped, slice_label, shard, other, out, transport, compute, trace=None,
                            gate=None, schedule=None):
    """Rank r's out = einsum of the gathered looped operand with its own ``other`` operand, computed
    as the Looped AllGather-Einsum ([Decomp] §5.1).

    Per local rank l: ``shard[l]`` is its shard of the looped operand (``looped`` = "lhs" or "rhs",
    sliced along ``slice_label``), ``other[l]`` its local operand, ``out[l]`` its output. Case 1
    (non-contracting m / n): DynamicUpdateSlice of the shard's rows / columns of out; case 2
    (contracting k): Addition into out (fp32); case 3 (batch b): DynamicUpdateSlice of its batches.
    ``schedule``: coco.SCHED_RING (default; unrolling by 2 is the same loop here, its double buffering
    being the chain's two receive buffers, [Decomp] §5.4.1) or coco.SCHED_BIDIRECTIONAL ([Decomp]
    §5.4.2: a prologue on the own shard, then each step receives shard r+k from one side and r-k from
    the other and computes both).
    ``trace`` (a list) makes every transfer carry its shard ID beside the data and receives
    (step, rank, shard_id) for each partial einsum. ``gate``: the four §5.5 times; when they say
    the loop does not pay, the original AllGather and one einsum run instead.
    """
    if looped not in ("lhs", "rhs") or slice_label not in "bmnk" or len(slice_label) != 1:
        raise ValueError("looped must be 'lhs' or 'rhs' and slice_label one of b, m, n, k")
    if slice_label == "n" and looped == "lhs" or slice_label == "m" and looped == "rhs":
        raise ValueError(f"{slice_label!r} is not a dimension of the {looped} operand")
    sched = coco.SCHED_RING if schedule is None else int(schedule)
    if sched not in (coco.SCHED_RING, coco.SCHED_UNROLL2, coco.SCHED_BIDIRECTIONAL):
        raise ValueError(f"unknown schedule {schedule!r}")
    n = transport.nranks
    L = transport.local_ranks
    sd = _dim(spec, looped, slice_label)
    ext = shard[0].shape[sd]
    if gate is not None and not decompose(gate):
        return _allgather_then_einsum(spec, looped, sd, shard, other, out, transport, compute)

    used = [0]  # partial einsums done (case 2: the first one writes out, the others add)

    def partial(held, sids, step):
        """The partial einsum of one shard per local rank: held[l] is shard sids[l] of the looped operand."""
        if trace is not None:
            trace.extend((step, r, sid) for r, sid in zip(L, sids))
        if slice_label == "k":  # case 2: DynamicSlice of the other operand along k, Addition
            od = _dim(spec, "rhs" if looped == "lhs" else "lhs", "k")
            oth = [o.narrow(od, sid * ext, ext) for o, sid in zip(other, sids)]
            if any(not t.is_contiguous() for t in oth):
                raise ValueError("case 2 needs the other operand's k slices contiguous (k its leading dimension)")
            lhs, rhs = (held, oth) if looped == "lhs" else (oth, held)
            if used[0] == 0:
                compute.einsum(spec, lhs, rhs, out)
            else:  # the Addition fused into the partial einsum (the shard in hand is not in flight)
                compute.einsum_accumulate(spec, lhs, rhs, out)
        else:
            od = spec.replace(" ", "").split("->")[1].index(slice_label)
            dst = [o.narrow(od, sid * ext, ext) for o, sid in zip(out, sids)]
            if slice_label == "b":  # case 3: DynamicSlice of the other operand along b
                ob = _dim(spec, "rhs" if looped == "lhs" else "lhs", "b")
                oth = [o.narrow(ob, sid * ext, ext) for o, sid in zip(other, sids)]
            else:
                oth = list(other)
            if any(not t.is_contiguous() for t in dst):
                raise ValueError("the DynamicUpdateSlice target must be contiguous (slice on a leading dimension)")
            lhs, rhs = (held, oth) if looped == "lhs" else (oth, held)
            compute.einsum(spec, lhs, rhs, dst)
        used[0] += 1

    orders = [coco.coco_shard_order(AG, sched if sched == coco.SCHED_BIDIRECTIONAL else coco.SCHED_RING, r, n)
              for r in L]
    own_ids = list(L) if trace is not None else None
    if sched != coco.SCHED_BIDIRECTIONAL:
        ch = _Chain(shard, 1, transport, own_ids)
        for i in range(n):
            sids = [o[i] for o in orders]
            h = ch.start() if i < n - 1 else None  # the shard in hand goes to r-1, r+1's arrives
            ch.check(sids, f"step {i}")
            partial(ch.cur, sids, i)
            if h is not None:
                ch.done(h)
        return out

    # bidirectional: the own shard, then one shard from each side per step
    left = _Chain(shard, 1, transport, own_ids)    # brings r+1, r+2, ...
    right = _Chain(shard, -1, transport, own_ids)  # brings r-1, r-2, ...
    pos = 0
    step = 0
    while pos < n:
        take = 1 if pos == 0 else min(2, n - pos)  # shards computed in this step
        after = pos + take
        # the next step takes shard r+(step+1) from the left and, if two remain, r-(step+1) from the right
        hl = left.start() if after < n else None
        hr = right.start() if n - after >= 2 else None
        if pos == 0:
            left.check([o[0] for o in orders], "prologue")
            partial(left.cur, [o[0] for o in orders], 0)
        else:
            left.check([o[pos] for o in orders], f"step {step} (left)")
            partial(left.cur, [o[pos] for o in orders], step)
            if take == 2:
                right.check([o[pos + 1] for o in orders], f"step {step} (right)")
                partial(right.cur, [o[pos + 1] for o in orders], step)
        if hl is not None:
            left.done(hl)
        if hr is not None:
            right.done(hr)
        pos = after
        step += 1
    return out


def _allgather_then_einsum(spec, looped, sd, shard, other, out, transport, compute):
    """The original operations: AllGather of the looped operand, then one einsum."""
    n = transport.nranks
    full_shape = list(shard[0].shape)
    full_shape[sd] *= n
    full = [torch.empty(full_shape, dtype=shard[0].dtype, device=shard[0].device) for _ in shard]
    chunks = [[torch.empty_like(shard[0]) for _ in range(n)] for _ in shard]
    transport.all_gather(list(shard), chunks)
    for c, f in zip(chunks, full):  # placed in partition order by the library's AllGather kernel
        compute.assemble(c, sd, f)
    lhs, rhs = (full, list(other)) if looped == "lhs" else (list(other), full)
    compute.einsum(spec, lhs, rhs, out)
    return out


# ------------------------------------------------ Looped Einsum-ReduceScatter


class _Acc:
    """An fp32 accumulator travelling around the ring (one chain of an Einsum-ReduceScatter): the tensor
    in hand on every local rank (added to in place), the buffer the next transfer lands in, and, in trace
    mode, the ID of the output shard it collects."""

    def __init__(self, bufs, shift, transport, trace_mode):
        self.acc, self.inc = bufs
        self.shift = shift
        self.t = transport
        self.ids = self.nid = None
        if trace_mode:
            dev = self.acc[0].device
            self.ids = [torch.zeros((1,), dtype=torch.int64, device=dev) for _ in self.acc]
            self.nid = [torch.empty_like(x) for x in self.ids]

    def start(self):  # CollectivePermuteStart
        h = self.t.permute(self.acc, self.inc, self.shift)
        hid = self.t.permute(self.ids, self.nid, self.shift) if self.ids is not None else None
        return h, hid

    def done(self, hs):  # CollectivePermuteDone
        h, hid = hs
        h.wait()
        self.acc, self.inc = self.inc, self.acc
        if hid is not None:
            hid.wait()
            self.ids, self.nid = self.nid, self.ids

    def tag(self, sids):
        if self.ids is not None:
            for x, s_ in zip(self.ids, sids):
                x.fill_(s_)

    def check(self, sids, what):
        if self.ids is not None:
            got = [int(x.item()) for x in self.ids]
            if got != list(sids):
                raise AssertionError(f"{what}: accumulators {got} in hand, schedule says {list(sids)}")


def looped_einsum_reduce_scatter(spec, lhs, rhs, out, transport, compute, trace=None, gate=None, schedule=None):
    """Rank r's out = shard r (rows of the LHS) of the sum over ranks q of lhs_q @ rhs_q, computed as
    the Looped Einsum-ReduceScatter ([Decomp] §5.1): fp32 accumulators travel the ring; each rank
    computes its partial for the shard ID of an accumulator while that accumulator is on its way, then
    adds it. ``schedule``:

    * coco.SCHED_RING (default): one accumulator {j -> j-1}; at iteration i rank q adds its partial for
      shard (q+i+1) mod N; output shard r collects the ranks r-1, r-2, ..., r.
    * coco.SCHED_UNROLL2 ([Decomp] §5.4.1): two interleaved chains travelling two hops per iteration,
      chain A collecting ranks r-1, r-3, ... and chain B ranks r-2, r-4, ...; each chain's Addition is
      fused into its partial einsum (coco_einsum_accumulate) and runs while the other chain travels; the
      chain that ends one hop short takes one more hop and rank r adds the two.
    The ring and bidirectional forms compute each partial while its accumulator is in flight and add
    it once the accumulator has arrived (the fused form would have to wait for the transfer first).
    * coco.SCHED_BIDIRECTIONAL ([Decomp] §5.4.2): a left-moving accumulator collects ranks r+a, ..., r+1
      and a right-moving one r-b, ..., r-1 (a = floor(N/2), b = floor((N-1)/2)); each takes one more hop
      onto rank r, which adds both to its own partial.

    ``out[l]``: fp32 [M/N, ...] per local rank. ``trace`` (a list): transfers carry shard IDs and the
    list receives (iteration, rank, shard_id) for the ring, (iteration, rank, "A" | "B", shard_id) for
    unroll-by-2 and (iteration, rank, "left" | "right", shard_id) for bidirectional. ``gate``: the four
    §5.5 times; when they say the loop does not pay, the original operations run: each rank's whole
    einsum, then a ReduceScatter of the results.
    """
    n = transport.nranks
    L = transport.local_ranks
    if out[0].dtype != torch.float32:
        raise ValueError("the accumulator (and so the output) of the distributed ReduceScatter is fp32")
    sched = coco.SCHED_RING if schedule is None else int(schedule)
    if sched not in (coco.SCHED_RING, coco.SCHED_UNROLL2, coco.SCHED_BIDIRECTIONAL):
        raise ValueError(f"unknown schedule {schedule!r}")
    md = _dim(spec, "lhs", "m")
    m = lhs[0].shape[md]
    if m % n:
        raise ValueError("the LHS rows do not split into equal shards")
    ms = m // n
    if gate is not None and not decompose(gate):
        return _einsum_then_reduce_scatter(spec, lhs, rhs, out, transport, compute)
    tmode = trace is not None
    part = [torch.empty_like(o) for o in out]

    def partial_into(dst, sids):
        """dst[l] = the partial einsum of local rank l for output shard sids[l] (its LHS rows of it)."""
        compute.einsum(spec, [x.narrow(md, s_ * ms, ms) for x, s_ in zip(lhs, sids)], list(rhs), dst)

    def step(chain, i, sids, label):
        """Iteration i of one chain whose transfer (if any) was started: its partial einsum (the first one
        straight into the accumulator, later ones into ``part`` for the Addition in finish)."""
        if i == 0:
            partial_into(chain.acc, sids)
            chain.tag(sids)
        else:
            partial_into(part, sids)

    def finish(chain, hs, i, sids, label):
        if i > 0:
            chain.done(hs)
            compute.accumulate(chain.acc, part)
        chain.check(sids, f"iteration {i}" + (f" ({label})" if label else ""))
        if tmode:
            trace.extend(((i, q, s_) if label is None else (i, q, label, s_)) for q, s_ in zip(L, sids))

    if sched == coco.SCHED_RING:
        # the accumulator changes buffers at every iteration after the first: start it in the buffer that
        # makes it end in ``out``
        other_buf = [torch.empty_like(o) for o in out]
        bufs = (list(out), other_buf) if n % 2 == 1 else (other_buf, list(out))
        A = _Acc(bufs, 1, transport, tmode)
        for i in range(n):
            sids = [(q + i + 1) % n for q in L]
            hs = A.start() if i > 0 else None
            step(A, i, sids, None)
            finish(A, hs, i, sids, None)
        for x, o in zip(A.acc, out):  # aligned at the loop end: each rank holds its own shard
            if x.data_ptr() != o.data_ptr():
                o.copy_(x)
        return out

    def new(shift):
        return _Acc(([torch.empty_like(o) for o in out], [torch.empty_like(o) for o in out]), shift, transport,
                    tmode)

    if sched == coco.SCHED_UNROLL2:
        # The two chains alternate so that each one's Addition, fused into its partial einsum (which needs
        # the accumulator to have arrived), runs while the other chain's accumulator is in flight: the
        # point of unrolling by 2 in [Decomp] §5.4.1.
        na, nb = (n + 1) // 2, n // 2
        A, B = new(2), new(2)

        def fused(chain, i, sids, label):
            compute.einsum_accumulate(spec, [x.narrow(md, s_ * ms, ms) for x, s_ in zip(lhs, sids)], list(rhs),
                                      chain.acc)
            chain.check(sids, f"iteration {i} ({label})")
            if tmode:
                trace.extend((i, q, label, s_) for q, s_ in zip(L, sids))

        def sids_a(i):
            return [(q + 1 + 2 * i) % n for q in L]

        def sids_b(i):
            return [(q + 2 + 2 * i) % n for q in L]

        step(A, 0, sids_a(0), "A")
        finish(A, None, 0, sids_a(0), "A")
        ha = A.start() if na > 1 else None
        if nb:
            step(B, 0, sids_b(0), "B")
            finish(B, None, 0, sids_b(0), "B")
        for i in range(1, na):
            A.done(ha)
            hb = B.start() if i < nb else None
            fused(A, i, sids_a(i), "A")  # while B travels
            ha = A.start() if i + 1 < na else None
            if i < nb:
                B.done(hb)
                fused(B, i, sids_b(i), "B")  # while A travels
        # epilogue: the chain whose last contribution came from rank r+1 takes one more hop
        if n % 2 == 0:
            A.shift = 1
            A.done(A.start())
        elif n > 1:
            B.shift = 1
            B.done(B.start())
        A.check(list(L), "after the epilogue (A)")
        if nb:
            B.check(list(L), "after the epilogue (B)")
            for l, o in enumerate(out):
                compute.fused_slice([A.acc[l], B.acc[l]], None, None, 0.0, 0, 0, o)
        else:
            for x, o in zip(A.acc, out):
                o.copy_(x)
        return out

    # bidirectional
    a_, b_ = n // 2, (n - 1) // 2
    left, right = new(1), new(-1)
    for i in range(max(a_, b_)):
        sl = [(q + i - a_) % n for q in L]
        sr = [(q + b_ - i) % n for q in L]
        hl = left.start() if 0 < i < a_ else None
        hr = right.start() if 0 < i < b_ else None
        if i < a_:
            step(left, i, sl, "left")
            finish(left, hl, i, sl, "left")
        if i < b_:
            step(right, i, sr, "right")
            finish(right, hr, i, sr, "right")
    if a_:
        left.done(left.start())
        left.check(list(L), "after the epilogue (left)")
    if b_:
        right.done(right.start())
        right.check(list(L), "after the epilogue (right)")
    partial_into(out, list(L))  # the own partial
    for l, o in enumerate(out):
        parts = [o] + ([left.acc[l]] if a_ else []) + ([right.acc[l]] if b_ else [])
        if len(parts) > 1:
            compute.fused_slice(parts, None, None, 0.0, 0, 0, o)  # own + left + right, in that order
    return out


def _einsum_then_reduce_scatter(spec, lhs, rhs, out, transport, compute):
    """The original operations: every rank's whole einsum (fp32), then a ReduceScatter onto the LHS rows
    (an all-to-all of the row shards, summed in rank order by the library's reduction kernel)."""
    n = transport.nranks
    L = transport.local_ranks
    shape = list(out[0].shape)
    full = [torch.empty([shape[0] * n] + shape[1:], dtype=torch.float32, device=out[0].device) for _ in L]
    compute.einsum(spec, list(lhs), list(rhs), full)
    S = out[0].numel()
    recv = [torch.empty(S * n, dtype=torch.float32, device=out[0].device) for _ in L]
    transport.all_to_all([f.reshape(-1) for f in full], recv)  # shard r of every rank's result to rank r
    for l, o in enumerate(out):
        compute.fused_slice([recv[l].narrow(0, s * S, S).view(o.shape) for s in range(n)], None, None, 0.0, 0, 0, o)
    return out


# ------------------------------------------------------ FusedAllReduce (split)


def fused_allreduce(partial, bias, residual, p, seed, out, transport, compute):
    """out = dropout(sum over ranks of partial + bias) + residual on every rank, as [CoCoNet]'s
    AllReduce Split + Fuse: each rank receives slice r (of N equal slices of the flattened tensor) of
    every rank's partial, sums them in rank order with the bias, dropout and residual of those elements
    only (whole-tensor element indices, so the mask is the one-device mask), and the finished slices
    are all-gathered. ``partial[l]``, ``residual[l]`` (or None), ``out[l]``: per local rank, one shape."""
    n = transport.nranks
    L = transport.local_ranks
    numel = partial[0].numel()
    vec = 16 // partial[0].element_size()
    if numel % (n * vec):
        raise ValueError(f"{numel} elements do not split into {n} slices of whole 16-byte vectors")
    S = numel // n
    H = partial[0].shape[-1]
    if bias is not None and S % H:
        raise ValueError("with a bias, every slice must hold whole rows of the last dimension")
    shape = (S // H, H) if S % H == 0 else (S,)  # the bias runs along the last dimension
    send = [x.reshape(-1) for x in partial]
    recv = [torch.empty(numel, dtype=partial[0].dtype, device=partial[0].device) for _ in L]
    transport.all_to_all(send, recv)  # ReduceScatter's data movement: slice r of every rank's partial
    mine = []
    for l, r in enumerate(L):
        o = torch.empty(S, dtype=out[0].dtype, device=out[0].device)
        res = None if residual is None else residual[l].reshape(-1).narrow(0, r * S, S).view(shape)
        got = [recv[l].narrow(0, s * S, S).view(shape) for s in range(n)]
        compute.fused_slice(got, bias, res, p, seed, r * S, o.view(shape))
        mine.append(o)
    dst = [[o.reshape(-1).narrow(0, s * S, S) for s in range(n)] for o in out]
    transport.all_gather(mine, dst)  # AllGather of the finished slices
    return out
