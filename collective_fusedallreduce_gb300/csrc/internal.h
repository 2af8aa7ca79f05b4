// Internal interfaces between the C-ABI layer (api.cu) and the kernels.
// Nothing here is exported from libcoco.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "coco.h"

namespace coco {

inline int dtype_size(int dt) { return dt == COCO_F32 ? 4 : 2; }

// ----------------------------------------------------------------- reductions

// Pointer tables of one reduction launch. Group g owns inputs
// in[g*nranks + r] and its distinct outputs out[g*nranks + j], j < nout[g].
struct ReduceTables {
  const void* in[COCO_MAX_PTRS];
  void* out[COCO_MAX_PTRS];
  int32_t nout[COCO_MAX_PTRS];
  const void* residual[COCO_MAX_PTRS];  // per group, or nullptr
};

// FusedAllReduce / AllReduce over `numel` elements per rank.
struct FarLaunch {
  ReduceTables t;
  int dtype;
  int nranks, ngroups;
  int64_t numel;
  const void* bias;  // nullptr = none
  int64_t bias_len;  // H
  bool dropout;
  uint32_t keep_threshold;  // keep iff hash >> 40 < keep_threshold
  float scale;
  uint64_t seed;
  uint64_t index_base;  // whole-tensor index of the first element (a multiple of the vector width)
};
cudaError_t launch_fused_allreduce(const FarLaunch& L, cudaStream_t s);

// ReduceScatter / AllGather over a tensor viewed as [outer, mid, inner] with
// the slice on `mid` (slice length mid / nranks). For reduce-scatter, `out`
// holds one pointer per (group, rank): rank r's slice. For all-gather, `in`
// holds one pointer per (group, rank) (rank s's slice) and `out` the distinct
// destinations of each group.
struct SliceLaunch {
  ReduceTables t;
  int dtype;
  int nranks, ngroups;
  int64_t outer, mid, inner;
};
cudaError_t launch_reduce_scatter(const SliceLaunch& L, cudaStream_t s);
cudaError_t launch_allgather(const SliceLaunch& L, cudaStream_t s);

// Scattered-tensor AllReduce over a device bucket table (header of 16 words,
// then 3 words per (bucket, rank) entry).
cudaError_t launch_scattered_allreduce(const void* table, int64_t nbuckets, int nranks, int dtype, float alpha,
                                       cudaStream_t s);

cudaError_t launch_keep_mask(uint64_t seed, uint32_t threshold, uint64_t first, uint64_t count,
                             uint8_t* mask, cudaStream_t s);

// ---------------------------------------------------------------- GEMM plans

// A dense row-major [nb][rows][cols] operand (elements).
struct View {
  const void* ptr;
  int32_t nb, rows, cols;
  int64_t ld, bstride;
};

// A dense row-major [nb][rows][cols] output (elements).
struct OutView {
  void* ptr;
  int64_t ld, bstride;
  int32_t nb, rows, cols;
};

// One contiguous K range of a job: the A operand is read at
// (batch a_b0+bb, rows a_r0 + i, k a_k0 + k), B at (batch b_b0+bb, k b_k0 + k,
// cols b_c0 + j), k < klen.
struct Seg {
  int16_t a, b;  // view indices
  int32_t a_b0, a_r0, a_k0;
  int32_t b_b0, b_k0, b_c0;
  int32_t klen;
};

// A block of output: batches [o_b0, o_b0+nb), rows [o_r0, o_r0+m), cols
// [o_c0, o_c0+n) of output `out`, the sum over segments seg0..seg0+nseg-1 in
// that order.
//
// With the FusedAllReduce epilogue the job's result is written to `nout`
// outputs (indices out .. out+nout-1, the distinct replicas of a group) and
// `res` is the replicated residual of the same shape (or null).
struct Job {
  int32_t out;
  int32_t o_b0, o_r0, o_c0;
  int32_t nb, m, n;
  int16_t seg0, nseg;
  int16_t nout;
  int16_t res_map;  // FusedAllReduce epilogue: index of the residual's tensor map in the launch (set there)
  int32_t kblocks;  // K blocks of the tile's whole segment loop (set by the tensor-core launcher)
  const void* res;
};

// The epilogue applied to every accumulator tile.
// EPI_ADD: out = out + accumulator, fp32 output (the Addition of the Looped CollectiveEinsum fused into
// the einsum); the job's `res` is its own output, read one strip ahead like the residual.
enum EpilogueMode { EPI_STORE = 0, EPI_FUSED_ALLREDUCE = 1, EPI_ADD = 2 };

// Pointwise part of the FusedAllReduce epilogue (bias over the last
// dimension, counter-hash dropout, then the residual), as in coco_fused_allreduce.
struct FarEpilogue {
  const void* bias = nullptr;  // [cols] of the output dtype, or null
  bool dropout = false;
  uint32_t keep_threshold = 1u << 24;
  float scale = 1.0f;
  uint64_t seed = 0;
};

struct GemmPlan {
  int in_dtype = COCO_BF16;
  int out_dtype = COCO_BF16;
  int mode = EPI_STORE;
  FarEpilogue far;
  std::vector<View> views;
  std::vector<OutView> outs;
  std::vector<Seg> segs;
  std::vector<Job> jobs;
};

// Tensor-core path (bf16 / f16 inputs, tcgen05 + TMA). Returns
// cudaErrorNotSupported if the plan violates a TMA rule the host checks.
cudaError_t launch_gemm_tc(const GemmPlan& plan, cudaStream_t s, unsigned int* err_word);
// The same in two steps: tc_prepare encodes the tensor maps and fills the
// parameter blocks (host only; *out is freed with tc_free), tc_launch
// enqueues them on `s` (any number of times; calls on one prepared plan must
// not run concurrently, as each sets the per-launch fields of its blocks).
struct TcPrepared;
cudaError_t tc_prepare(const GemmPlan& plan, TcPrepared** out);
cudaError_t tc_launch(TcPrepared* prep, cudaStream_t s, unsigned int* err_word);
void tc_free(TcPrepared* prep);
// fp32 path (FMA units).
cudaError_t launch_gemm_simt(const GemmPlan& plan, cudaStream_t s);

// Device error word of the GEMM kernels (bounded waits record here).
unsigned int* gemm_error_word();
// One CTA waits on a barrier nothing completes, bounded by timeout_ns (the failure-path self-test).
cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t s, unsigned int* err_word);

int sm_count();

// Counts one kernel launch (exported as coco_kernel_launches).
void count_launch();

}  // namespace coco
