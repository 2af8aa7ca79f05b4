/*
 * coco.h -- C interface of libcoco: collectives fused with, and decomposed
 * around, their dependent computation, for N logical ranks whose buffers all
 * live in the memory of one GPU (sm_103a).
 *
 * Sources (cited by title and section):
 *   [CoCoNet] "Breaking the Computation and Communication Abstraction Barrier
 *             in Distributed Machine Learning Workloads" (ASPLOS '22).
 *   [Decomp]  "Overlap Communication with Dependent Computation via
 *             Decomposition in Large Deep Learning Models" (ASPLOS '23).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors. A coco_tensor describes one distributed tensor in [CoCoNet]'s
 * layout terms (the tensor-layout description accompanying its Fig. 3):
 *   COCO_SLICED     equally split along `slice_dim` over the ranks; rank r
 *                   holds slice r. `shape` is the GLOBAL shape and
 *                   shape[slice_dim] must divide by `nranks`.
 *   COCO_REPLICATED the same values on every rank. `shape` is the per-rank
 *                   shape. An input is read from ptr[g*nranks + 0] only; an
 *                   output is written to every DISTINCT pointer of the group
 *                   (pass one pointer nranks times to get one copy).
 *   COCO_LOCAL      same shape, different values on every rank. `shape` is the
 *                   per-rank shape.
 * `ngroups` independent groups of `nranks` ranks each (the subgroups of a 2-D
 * device mesh, [Decomp] §2.2 Fig. 3) share one call; pointers are group-major:
 * ptr[g*nranks + r] is rank r of group g.
 *
 * Memory. Every pointer is a device pointer owned by the caller; each rank's
 * buffer is dense and row-major. The library allocates no device memory; its
 * own state is fixed-size device globals (an error word, and arrival counters
 * for tensor-core launches whose CTAs wait on one another; up to 1024 such
 * launches may be in flight at once).
 * Device pointers must be 16-byte aligned and the innermost per-rank
 * dimension a multiple of 8 elements, else COCO_ERR_ALIGN.
 *
 * Streams. `stream` is a cudaStream_t (NULL = the legacy default stream).
 * Every call validates its arguments on the host, returns an error before any
 * CUDA call if they are invalid, and otherwise enqueues its kernels on
 * `stream` and returns without synchronising. All N ranks of all groups are
 * processed by the one call.
 *
 * Threads. Calls may come from several host threads at once: a call's host
 * state is its own, the caches the library sets up once (kernel attributes,
 * SM counts, device addresses) are atomic or locked, and
 * coco_last_cuda_error() is per thread.
 *
 * CUDA graphs. Because no call synchronises or allocates, a sequence of calls
 * may be captured into a CUDA graph (stream capture) and replayed; a replay
 * repeats the launches with the pointers and sizes of the capture. A captured
 * tensor-core launch whose CTAs wait on one another keeps the arrival counter
 * it was given at capture (reset by a memset node before it), so two
 * instantiations of one such graph must not run at the same time; launches of
 * one instantiated graph are ordered behind each other by CUDA.
 *
 * Aliasing. An output may not overlap any input, except where an entry point
 * says otherwise; violations return COCO_ERR_ALIAS.
 *
 * Errors. The return value is the only error channel. COCO_ERR_CUDA means a
 * launch failed (the CUDA error is kept: coco_last_cuda_error()). Device-side
 * waits are bounded; a wait that gives up records COCO_ERR_TIMEOUT, which
 * coco_device_status() reports.
 *
 * Empty tensors (a zero in any extent) are valid: the call returns COCO_OK
 * and launches nothing.
 */
#ifndef COCO_H_
#define COCO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  COCO_OK = 0,
  COCO_ERR_NULL = 1,        /* a required pointer is NULL */
  COCO_ERR_SHAPE = 2,       /* shapes or rank counts disagree, or a slice is uneven */
  COCO_ERR_DTYPE = 3,       /* unknown dtype, or operand dtypes disagree */
  COCO_ERR_LAYOUT = 4,      /* an operand has a layout the operation does not take */
  COCO_ERR_ALIGN = 5,       /* pointer not 16-byte aligned, or inner dim not a multiple of 8 */
  COCO_ERR_ALIAS = 6,       /* an output overlaps an input or another output */
  COCO_ERR_UNSUPPORTED = 7, /* valid request outside what this library implements */
  COCO_ERR_CUDA = 8,        /* a CUDA runtime call or kernel launch failed */
  COCO_ERR_TIMEOUT = 9,     /* a bounded device-side wait gave up */
  COCO_ERR_VALUE = 10       /* a scalar argument is out of range (e.g. dropout p) */
} coco_status;

typedef enum { COCO_F32 = 0, COCO_F16 = 1, COCO_BF16 = 2 } coco_dtype;

typedef enum { COCO_LOCAL = 0, COCO_SLICED = 1, COCO_REPLICATED = 2 } coco_layout;

#define COCO_MAX_PTRS 64 /* ngroups * nranks <= COCO_MAX_PTRS */
#define COCO_MAX_DIMS 3

typedef struct {
  int32_t dtype;                 /* coco_dtype */
  int32_t layout;                /* coco_layout */
  int32_t ndim;                  /* 1..COCO_MAX_DIMS */
  int32_t slice_dim;             /* COCO_SLICED only: the sliced dimension */
  int64_t shape[COCO_MAX_DIMS];  /* global shape if SLICED, per-rank shape otherwise */
  int32_t nranks;                /* ranks per group, 1..COCO_MAX_PTRS */
  int32_t ngroups;               /* independent groups, >= 1 */
  void* ptr[COCO_MAX_PTRS];      /* device pointers, ptr[g*nranks + r] */
} coco_tensor;

/* ------------------------------------------------------------------ fused */

/*
 * FusedAllReduce ([CoCoNet] §5.2 and the AllReduce Fuse transformation;
 * the computation of its Fig. 3, lines 9-13):
 *
 *   out_q[e] = dropout( sum_{r=0}^{N-1} partials_r[e] + bias[e mod H] ) + residual[e]
 *
 * for every rank q of every group, with the sum, bias, dropout scale and
 * residual in fp32 registers and one rounding to the output type at the
 * store; the summed value is never written to memory.
 *
 *   partials  LOCAL, dtype T in {F32, F16, BF16}, any per-rank shape S.
 *   bias      device pointer to H = S[ndim-1] elements of T, or NULL.
 *   residual  REPLICATED, dtype T, shape S, or NULL (read from rank 0's pointer).
 *   dropout_p probability of dropping, in [0, 1]; 0 disables dropout.
 *   seed      dropout seed. Element e (0-based row-major index inside one
 *             rank's tensor, the same on every rank and group) is kept iff
 *             (splitmix64(seed, e) >> 40) < floor((1 - p) * 2^24), where
 *             splitmix64(seed, e) is the (e+1)-th output of SplitMix64
 *             started at state `seed`; kept values are multiplied by
 *             (float)(1 / (1 - p)) and dropped ones become 0 before the
 *             residual is added. Bit-exact: see coco_dropout_keep_mask.
 *   out       REPLICATED, dtype T, shape S. out_q may equal partials_q or the
 *             residual pointer exactly (in place); any other overlap is
 *             COCO_ERR_ALIAS.
 */
coco_status coco_fused_allreduce(const coco_tensor* partials, const void* bias,
                                 const coco_tensor* residual, float dropout_p, uint64_t seed,
                                 const coco_tensor* out, void* stream);

/*
 * The same FusedAllReduce over a contiguous part of larger tensors, for the
 * chunked form of [CoCoNet]'s Overlap construct (§5.3, Fig. 9: the AllReduce
 * of a chunk runs while the MatMul produces the next one). index_base is the
 * row-major index, inside one rank's whole tensor, of the first element of
 * the part passed; dropout element indices and the bias phase continue from
 * it, so calls over consecutive parts give, bit for bit, the result of one
 * coco_fused_allreduce over the whole. index_base must be a multiple of
 * 16 / sizeof(T) elements (else COCO_ERR_ALIGN); coco_fused_allreduce is
 * index_base = 0. Everything else as coco_fused_allreduce.
 */
coco_status coco_fused_allreduce_at(const coco_tensor* partials, const void* bias,
                                    const coco_tensor* residual, float dropout_p, uint64_t seed,
                                    uint64_t index_base, const coco_tensor* out, void* stream);

/*
 * Plain AllReduce ([Decomp] §2.1): out_q = sum_r in_r (fp32 sum in rank order
 * 0..N-1, one rounding), for every rank q. in LOCAL, out REPLICATED, same
 * dtype and shape. In place (out_q == in_q exactly) is allowed.
 */
coco_status coco_allreduce(const coco_tensor* in, const coco_tensor* out, void* stream);

/*
 * ReduceScatter ([Decomp] §2.1): rank r receives slice r (along
 * out->slice_dim) of sum_q in_q, summed in fp32 in rank order 0..N-1.
 * in LOCAL with per-rank shape S; out SLICED with global shape S.
 */
coco_status coco_reduce_scatter(const coco_tensor* in, const coco_tensor* out, void* stream);

/*
 * AllGather ([Decomp] §2.1): every rank receives the concatenation, in
 * partition-ID order along in->slice_dim, of all ranks' slices. in SLICED with
 * global shape S; out REPLICATED with shape S. A bit-exact copy.
 */
coco_status coco_allgather(const coco_tensor* in, const coco_tensor* out, void* stream);

/*
 * AllReduce Split RS-AG ([CoCoNet], split transformation): a ReduceScatter of
 * `in` into `scratch` (the sliced intermediate) followed by an AllGather of
 * `scratch` into `out`. in LOCAL shape S; scratch SLICED global shape S (the
 * caller's memory; slice_dim chooses the split); out REPLICATED shape S.
 * Bit-identical to coco_allreduce (both sum in fp32 in rank order).
 */
coco_status coco_allreduce_rs_ag(const coco_tensor* in, const coco_tensor* scratch,
                                 const coco_tensor* out, void* stream);

/*
 * AllReduce Split RS-AG for callers that cannot allocate device memory. The
 * pages have no counterpart of this entry point; it exists for code that may
 * not call cudaMalloc once running (a latency-critical loop where an
 * allocation could stall or fail mid-step, or a plug-in inside an application
 * that owns all device memory). Same result as coco_allreduce_rs_ag (in LOCAL,
 * out REPLICATED, same dtype and shape), but the sliced intermediate lives in
 * a fixed 16 MiB array inside libcoco that every GPU loading the library
 * holds until the process exits, split on dimension 0.
 *   - A call needs ngroups * numel * element-size bytes (plus per-slice
 *     rounding to 256 bytes); larger requests return COCO_ERR_UNSUPPORTED
 *     before any CUDA call.
 *   - Extents follow the library's usual rule (each dimension and the
 *     per-rank element count at most 2^40, else COCO_ERR_SHAPE), checked
 *     before any size is multiplied.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address with cudaGetSymbolAddress and caches it for the
 *     current CUDA context; a call in a new context (after cudaDeviceReset,
 *     say) looks it up again. Make the first call in a context before any
 *     stream capture: a call that needs the look-up while `stream` is being
 *     captured returns COCO_ERR_UNSUPPORTED and launches nothing.
 *   - All calls share the array and it keeps the last call's contents
 *     (nothing needs to start at zero: the ReduceScatter writes every element
 *     the AllGather reads). Calls whose kernels can overlap on the GPU race on
 *     it; calls ordered on one stream do not.
 *   - It allocates nothing (no cudaMalloc, no cudaFree, no allocating
 *     library routine).
 */
coco_status coco_allreduce_rs_ag_noalloc(const coco_tensor* in, const coco_tensor* out, void* stream);

/* ------------------------------------------------------ scattered tensors */

/*
 * AllReduce of scattered tensors ([CoCoNet], the section on scattered
 * tensors): the gradients of data parallelism live in many separate buffers;
 * one kernel reduces all of them without first copying them into one buffer.
 * Each tensor is cut into buckets of at most 1024 elements, and each bucket is
 * described per rank by 12 bytes: the 64-bit address of the rank's tensor and
 * a 32-bit offset. Warps take buckets round-robin.
 *
 * The bucket table is built once (the same tensors are reduced every training
 * step) into caller-owned device memory of coco_scattered_table_bytes() bytes:
 * a 64-byte header, then nbuckets * nranks entries of 12 bytes, rank-inner. An
 * entry's 32-bit offset holds the bucket index within its tensor in bits
 * 10..31 (the element offset is that index * 1024) and the bucket length - 1
 * in bits 0..9.
 */
typedef struct {
  void* table;       /* device table (caller's memory) */
  int64_t nbuckets;  /* buckets over all tensors */
  int32_t nranks;
  int32_t dtype;     /* coco_dtype of every tensor */
} coco_scattered_plan;

/* Bytes of device memory the table of these tensors needs (64 + 12 * nbuckets * nranks). */
size_t coco_scattered_table_bytes(int32_t ntensors, const int64_t* numels, int32_t nranks);

/*
 * Builds the table into `table` (device, 16-byte aligned, at least
 * coco_scattered_table_bytes() bytes; a host-to-device copy ordered on
 * `stream`) and fills `plan`. `tensors[r * ntensors + t]` is rank r's tensor t
 * (device pointer, 16-byte aligned, numels[t] elements of `dtype`, dense);
 * numels[t] < 2^32. Tensors may not overlap each other or the table
 * (COCO_ERR_ALIAS). The upload reads a host buffer that lives only during the
 * call, so a call on a stream under capture returns COCO_ERR_UNSUPPORTED (build
 * the table first; the AllReduce itself may be captured).
 */
coco_status coco_scattered_table_build(int32_t ntensors, const int64_t* numels, int32_t dtype, int32_t nranks,
                                       void* const* tensors, void* table, size_t table_bytes,
                                       coco_scattered_plan* plan, void* stream);

/*
 * In place on every rank: tensor_r[t][e] = alpha * sum_{q=0}^{N-1} tensor_q[t][e]
 * for every tensor t, with the sum and the scale in fp32 (rank order 0..N-1)
 * and one rounding; alpha = 1 is the plain AllReduce, 1/N averages.
 */
coco_status coco_scattered_allreduce(const coco_scattered_plan* plan, float alpha, void* stream);

/* ---------------------------------------------------------------- einsums */

/*
 * Supported specs: "mk,kn->mn" (2-D operands) and "bmk,bkn->bmn" (3-D).
 * Operand storage: lhs row-major [.., m, k], rhs row-major [.., k, n], out
 * row-major [.., m, n]. lhs and rhs share a dtype; BF16 and F16 run on the
 * tensor cores with fp32 accumulation; F32 runs on fp32 FMA units. The output
 * dtype is out->dtype (F32, F16 or BF16), rounded once from the fp32
 * accumulator.
 *
 * Tensor-core limit: the loop that produces one output region (its K-segments:
 * the N rank slices of case 2, of the Einsum-ReduceScatter and of the fused
 * MatMul) must fit one launch's parameter block, at most 80 distinct operand
 * views (two per rank slice, so N <= 40 for those forms) and 192 K-segments.
 * Larger requests return COCO_ERR_UNSUPPORTED before anything is launched.
 */

/*
 * Local MatMul ([CoCoNet] Fig. 3 line 7 and its layout rule: MatMul of two
 * tensors sliced on the contracting dimension yields a local tensor):
 * out_r = lhs_r @ rhs_r for every rank. lhs: LOCAL, or SLICED on k; rhs:
 * LOCAL or REPLICATED, or SLICED on k; out: LOCAL (per-rank shape).
 */
coco_status coco_einsum(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                        const coco_tensor* out, void* stream);

/*
 * out_r += lhs_r @ rhs_r for every rank r, with the addition done in the einsum's epilogue: each output
 * element is read once, added to the fp32 accumulator and written once (the Addition update of the
 * Looped CollectiveEinsum fused into the partial einsum, [Decomp] §5.1 and the loop of §5.4.1; used by
 * the one-rank-per-device loops, where an accumulator or a case-2 output grows by one partial each
 * iteration). Operands as coco_einsum; `out` is LOCAL, fp32 (else COCO_ERR_DTYPE), read and written in
 * place, and may not overlap an operand (COCO_ERR_ALIAS). A contraction of length 0 leaves `out` as it
 * is. fp32 operands run on the FMA path.
 */
coco_status coco_einsum_accumulate(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                   const coco_tensor* out, void* stream);

/*
 * MatMul fused with FusedAllReduce ([CoCoNet] Fig. 3 lines 7-13; the
 * overlap of its MatMul with the AllReduce, §5.3 / Fig. 9, taken to a single
 * kernel on one GPU):
 *
 *   out_q = dropout( sum_{r=0}^{N-1} lhs_r @ rhs_r + bias ) + residual
 *
 * for every rank q of every group. lhs SLICED on k (per rank [m, k/N]); rhs
 * SLICED on k (per rank [k/N, n]); lhs and rhs F16 or BF16 (the same);
 * out REPLICATED [m, n], F16 or BF16; bias, residual, dropout_p and seed as in
 * coco_fused_allreduce (same dtype as out; element index e = row * n + col).
 * The sum over ranks accumulates in fp32 on the tensor cores (rank order
 * 0..N-1) and is never written to memory: no per-rank partial exists. out_q
 * may equal the residual pointer exactly; outputs may not overlap lhs, rhs or
 * bias, and a buffer may be a replica of one group only (else COCO_ERR_ALIAS).
 * A zero contraction length returns COCO_ERR_UNSUPPORTED; F32 operands or
 * output return COCO_ERR_UNSUPPORTED.
 */
coco_status coco_matmul_fused_allreduce(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                        const void* bias, const coco_tensor* residual, float dropout_p,
                                        uint64_t seed, const coco_tensor* out, void* stream);

/*
 * Looped AllGather-Einsum ([Decomp] §4 Fig. 4 and §5.1, Alg. 1): exactly one
 * operand is SLICED (the looped operand); the other is LOCAL or REPLICATED
 * (the local operand). Rank r computes, for i = 0..N-1 in this order, the
 * partial einsum with shard s = (r + i) mod N of the looped operand (the
 * shard it holds after i CollectivePermutes along {j -> j-1}), and updates
 * the result:
 *   looped operand sliced on a non-contracting dim (m of lhs / n of rhs):
 *       case 1, DynamicUpdateSlice of the shard's rows / columns;
 *   sliced on the contracting dim k: case 2, the local operand is
 *       DynamicSliced along k and the Update is an Addition (accumulated in
 *       fp32 across all N steps, stored once);
 *   sliced on the batch dim b: case 3, the local operand is DynamicSliced
 *       along b and the result DynamicUpdateSliced along b.
 * out: LOCAL with the full (gathered) per-rank result shape, or REPLICATED if
 * the local operand is REPLICATED.
 */
coco_status coco_looped_ag_einsum(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                  const coco_tensor* out, void* stream);

/*
 * Looped Einsum-ReduceScatter ([Decomp] §4 Fig. 5 and §5.1): lhs and rhs are
 * both SLICED on the contracting dimension k (so each rank's product is a
 * local partial sum); out is SLICED on m (lhs is DynamicSliced) or n (rhs is
 * DynamicSliced), with the global result shape. Output shard r is
 *     y_r = sum over q = r-1, r-2, ..., r (mod N) of (lhs_q @ rhs_q)[shard r],
 * the ring order in which the accumulated shard travels {j -> j-1} so that
 * its ID equals the partition ID at the loop end, accumulated in fp32 and
 * stored once.
 */
coco_status coco_looped_einsum_rs(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                  const coco_tensor* out, void* stream);

/*
 * Shard schedules of the Looped CollectiveEinsum ([Decomp] §5.4). They change
 * only the order in which shards are visited (AllGather) or partials are
 * collected (ReduceScatter), i.e. the fp32 accumulation order; the result is
 * the same einsum.
 *   COCO_SCHED_RING          §5.1: permutes {j -> j-1}. AllGather: rank r visits
 *                            r, r+1, ..., r-1; ReduceScatter: output shard r
 *                            collects ranks r-1, r-2, ..., r.
 *   COCO_SCHED_UNROLL2       §5.4.1 (loop unrolled by 2): ReduceScatter as two
 *                            interleaved chains travelling two hops per step,
 *                            r-1, r-3, ... then r-2, r-4, ..., summed in an
 *                            epilogue. On one GPU the AllGather order is the ring
 *                            order (unrolling there only removes copies).
 *   COCO_SCHED_BIDIRECTIONAL §5.4.2: shards / accumulators travel both ways.
 *                            AllGather: r, r+1, r-1, r+2, r-2, ...;
 *                            ReduceScatter: r+a, ..., r+1 (left-moving), then
 *                            r-b, ..., r-1 (right-moving), then r itself, with
 *                            a = floor(N/2), b = floor((N-1)/2).
 */
typedef enum { COCO_SCHED_RING = 0, COCO_SCHED_UNROLL2 = 1, COCO_SCHED_BIDIRECTIONAL = 2 } coco_schedule;

/* coco_looped_ag_einsum with an explicit schedule (a coco_schedule value; others: COCO_ERR_VALUE). */
coco_status coco_looped_ag_einsum_sched(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                        const coco_tensor* out, int schedule, void* stream);

/* coco_looped_einsum_rs with an explicit schedule (a coco_schedule value; others: COCO_ERR_VALUE). */
coco_status coco_looped_einsum_rs_sched(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                        const coco_tensor* out, int schedule, void* stream);

/*
 * The shard schedule the looped entry points follow, for callers that run the
 * loop themselves (one rank per process, the permutes over a network):
 *   kind 0 (AllGather-Einsum):  order[i] = the shard rank `rank` computes on at
 *                               step i;
 *   kind 1 (Einsum-ReduceScatter): order[i] = the rank whose partial output
 *                               shard `rank` receives at step i (the fp32
 *                               accumulation order).
 * [Decomp] §5.1 (ring) and §5.4 (unroll-by-2, bidirectional); see
 * coco_schedule. `order` is a host array of `nranks` int32 (caller-owned).
 * nranks in 1..COCO_MAX_PTRS and 0 <= rank < nranks, else COCO_ERR_SHAPE;
 * unknown kind or schedule: COCO_ERR_VALUE; NULL order: COCO_ERR_NULL.
 * Host only; no CUDA call.
 */
coco_status coco_shard_order(int32_t kind, int32_t schedule, int32_t rank, int32_t nranks, int32_t* order);

/*
 * The cost model that enables the decomposition ([Decomp] §5.5, "cost model
 * and enabling mechanism"): an AllGather-Einsum or Einsum-ReduceScatter is
 * replaced by its Looped CollectiveEinsum only when it is expected to pay,
 *     orig_comp + orig_comm >= max(orig_comp, ring_comm) + epilogue_cost,
 * where orig_comp and orig_comm are the times of the original einsum and
 * collective, ring_comm the time of the CollectivePermutes along the logical
 * ring, and epilogue_cost the time of the prologue or epilogue the schedule
 * adds (all in one unit). Writes 1 (decompose) or 0 (keep the original
 * operations) to *profitable. Every time must be finite and >= 0, else
 * COCO_ERR_VALUE (and *profitable is untouched); NULL: COCO_ERR_NULL. Host
 * only; no CUDA call.
 */
coco_status coco_loop_profitable(double orig_comp, double orig_comm, double ring_comm, double epilogue_cost,
                                 int32_t* profitable);

/* ------------------------------------------------------------- utilities */

/*
 * Writes mask[i] = 1 if element (first_index + i) is kept by the dropout of
 * coco_fused_allreduce with (seed, dropout_p), else 0, for i < count.
 * `mask` is a device pointer to `count` bytes (no alignment rule). Computed by
 * the same device code as the fused kernel; for bit-exact comparison.
 */
coco_status coco_dropout_keep_mask(uint64_t seed, float dropout_p, uint64_t first_index,
                                   uint64_t count, uint8_t* mask, void* stream);

/*
 * Synchronises `stream`, then reports and clears the device-side error word
 * (COCO_ERR_TIMEOUT if a bounded wait in a kernel gave up since the last
 * call). Returns COCO_ERR_CUDA if the synchronisation itself fails.
 */
coco_status coco_device_status(void* stream);

/*
 * Self-test of the device-side failure path (no counterpart on the pages):
 * one CTA allocates tensor memory, then one warp waits on an mbarrier phase
 * that nothing completes, with the bounded wait the tensor-core kernels use but
 * a limit of timeout_ns (1e3 .. 1e9 ns, else COCO_ERR_VALUE) on %globaltimer.
 * When the limit passes, the kernel records COCO_ERR_TIMEOUT and raises its
 * abort flag, the owner frees the tensor memory, and every thread returns: the
 * next coco_device_status() reports COCO_ERR_TIMEOUT (once) and the context
 * stays usable. Nothing faults, traps or hangs.
 */
coco_status coco_wait_selftest(uint64_t timeout_ns, void* stream);

/*
 * Number of kernels this library has launched in this process so far (all
 * threads, all devices). Launch accounting for benchmarks and tests.
 */
uint64_t coco_kernel_launches(void);

/*
 * Plan cache of the einsum entry points (coco_einsum, coco_einsum_accumulate, coco_matmul_fused_allreduce,
 * coco_looped_ag_einsum[_sched], coco_looped_einsum_rs[_sched]). A call whose
 * arguments repeat an earlier valid call's exactly (entry point, spec,
 * schedule, every in-use field of every coco_tensor including its pointers,
 * bias pointer, dropout_p, seed, and the current device) reuses that call's
 * plan and encoded tensor maps, skipping host validation and planning; the
 * stream may differ. Up to 64 plans are kept (least recently used dropped),
 * in host memory only. Freeing a buffer and passing a new one at the same
 * address with the same shape is safe: a plan depends only on the keyed
 * values. Counters are cumulative for the process; clear() drops every plan
 * (not the counters). Both are thread-safe; NULL arguments are skipped.
 */
void coco_plan_cache_stats(uint64_t* hits, uint64_t* misses, uint64_t* entries);
void coco_plan_cache_clear(void);

/* The cudaError_t (as int) of the most recent COCO_ERR_CUDA on this thread. */
int coco_last_cuda_error(void);

/* A static, human-readable name for a status code. */
const char* coco_status_string(coco_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int coco_version(void);

#ifdef __cplusplus
}
#endif

#endif /* COCO_H_ */
