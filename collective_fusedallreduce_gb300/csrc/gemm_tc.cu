// Tensor-core GEMM for sm_103a (tcgen05 + TMEM + TMA), driven by a plan of
// jobs and K-segments so one persistent launch runs every rank's part of a
// Looped CollectiveEinsum.
//
// [Decomp] "Overlap Communication with Dependent Computation via
// Decomposition in Large Deep Learning Models", §5.1 (Looped
// CollectiveEinsum, Alg. 1): on one GPU a CollectivePermute of a shard is a
// read of that shard where it lives, so the loop over shards becomes the
// order of K-segments (Addition: accumulated in TMEM) or of output jobs
// (DynamicUpdateSlice: the epilogue's row / column / batch offset).
//
// Kernel shape (one CTA per SM, CTA pairs in clusters of two, persistent
// over work units of two vertically adjacent 128 x 256 output tiles):
//   warp 0      TMA producer: per k-block (64 deep) an A tile [128 x 64]
//               (K-major, 128B swizzle) and B columns (N-major, 64-column
//               boxes, 128B swizzle) into an mbarrier ring of stages.
//   warp 1      allocates 512 TMEM columns (two fp32 128 x 256 accumulators)
//               and issues tcgen05.mma from one elected lane: either one
//               M=128, N=256 MMA per CTA, each CTA loading its own A tile and
//               the whole B tile (4 stages of 48 KB), or, for long k-loops, one
//               M=256 MMA over both CTAs (tcgen05 cta_group::2, 6 stages of
//               32 KB per CTA). No copy writes into another CTA's shared memory.
//   warps 2..5  epilogue, one TMEM lane quarter each: tcgen05.ld 32 lanes x
//               32 columns, convert (or, for the FusedAllReduce, add bias,
//               apply dropout and add the residual), stage a 128-byte-wide
//               swizzled strip in shared memory and bulk-store it by TMA;
//               tiles that overhang their job's region use bounded 16-byte
//               stores instead.
// Every mbarrier wait is bounded by %globaltimer; on expiry the kernel records
// COCO_ERR_TIMEOUT in the error word, raises an abort flag for the other
// roles, drains its own outstanding copies / MMAs (bounded again), frees TMEM
// and returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace coco {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BOX_BYTES = BK * 64 * 2;         // 8 KB (64 k-rows x 128 B)
constexpr int B_BYTES = B_BOX_BYTES * (BN / 64);  // 32 KB
constexpr int EPI_STRIP = 32 * 128;                 // one strip: 32 rows x 128 B

// Shared-memory budget. ONE CTA PER MMA (TWO_SM = false): each CTA of a pair
// loads its A tile and the whole B tile into its own shared memory, 48 KB per
// stage, 4 stages. TWO_SM: the pair runs one M=256 MMA over both CTAs'
// shared memory (tcgen05 cta_group::2), each CTA holding its own A tile and
// its own 128-column half of B, 32 KB per stage, 6 stages. Four epilogue
// warps (one per TMEM lane quarter) in both.
//
// The FusedAllReduce epilogue keeps the same depth of stages: each epilogue
// warp has one output strip and one residual strip, which the next chunk's
// residual is loaded into by TMA (one mbarrier per warp) while the current one
// is computed. Its output strip is rewritten only once the previous chunk's
// bulk stores (one per replica) have read it; its tiles have long K loops, so
// the epilogue has the time, and the operand ring keeps its sixth stage
// (2-3 % faster than two output strips and five stages).
template <int MODE, bool TWO_SM>
struct Cfg {
  static constexpr int B_STAGE = TWO_SM ? B_BYTES / 2 : B_BYTES;
  static constexpr int STAGE = A_BYTES + B_STAGE;
  static constexpr int STAGES = TWO_SM ? 6 : 4;
  static constexpr int EPI_WARPS = 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int EPI_OFF = STAGES * STAGE;
  static constexpr int STRIPS = 2;  // two output strips; FusedAllReduce: one output strip and the residual strip
  static constexpr int BAR_OFF = EPI_OFF + EPI_WARPS * STRIPS * EPI_STRIP;
  // full, empty, tmem full x2, tmem empty x2, drain (+ one residual barrier per epilogue warp)
  static constexpr int NUM_BARS = 2 * STAGES + 5 + (MODE == 0 ? 0 : EPI_WARPS);
  static constexpr int SMEM_BYTES = BAR_OFF + 8 * NUM_BARS + 16 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
};
// The pair MMA needs fewer operand bytes per SM and a deeper ring, which pays
// when tiles have long K loops (operand-bound); with short ones the epilogue
// dominates and the two CTAs are better left independent.
constexpr int kTwoSmMinKBlocks = 4;
constexpr uint32_t TMEM_COLS = 512;
constexpr int GROUP_M = 16;  // tile rasterisation for large B operands: 16 m-tiles per group, n-major inside
constexpr uint64_t kTimeoutNs = 2000000000ull;

constexpr int MAX_MAPS = 80;
constexpr int MAX_JOBS = 128;
constexpr int MAX_SEGS = 192;
constexpr int MAX_OUTS = 32;

struct TcParams {
  CUtensorMap maps[MAX_MAPS];
  CUtensorMap omaps[MAX_OUTS];  // output maps: box {128 bytes of columns, 32 rows, 1}
  Job jobs[MAX_JOBS];
  Seg segs[MAX_SEGS];
  OutView outs[MAX_OUTS];
  int32_t unit_start[MAX_JOBS + 1];  // first work unit (a pair of vertically adjacent tiles) of each job
  int32_t njobs;
  int32_t group_pairs;  // rasterisation: pairs of m-tiles per group, n-major inside a group
  int32_t wave_sync;    // producers wait for each other between waves (cooperative launches only)
  unsigned int* wave_counter;  // this launch's arrival counter (zeroed before the launch)
  int32_t total_units;
  uint32_t idesc;
  int32_t out_dtype;
  unsigned int* err;
  // FusedAllReduce epilogue (EPI_FUSED_ALLREDUCE only; EPI_ADD uses none of it)
  const void* bias;
  uint64_t seed;
  uint32_t keep_threshold;
  float scale;
  int32_t dropout;
};
static_assert(sizeof(TcParams) <= 32000, "kernel parameter block too large");

// ------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait. Returns false on timeout or when another role aborted.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            uint64_t timeout_ns = kTimeoutNs) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 31) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > timeout_ns) return false;
    }
  }
}
// The common case (phase already complete) stays inline.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_test(bar, parity) || mbar_wait_slow(bar, parity, abort_flag);
}
// The same for a whole warp, with one answer for all its lanes. Only lane 0
// polls a phase that is not complete yet; the lanes that issue async
// operations afterwards are lane 0 (the elected lane of a converged warp).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               uint64_t timeout_ns = kTimeoutNs) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_slow(bar, parity, abort_flag, timeout_ns);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}
// One lane of a converged warp (the lowest), chosen by the hardware.
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, e;\n\t}"
      : "=r"(p));
  return p != 0;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Bulk tensor store of one 32-row strip; completion tracked per thread in bulk groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// At most one committed bulk group may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The shared::cluster address of the same shared-memory offset in CTA 0 of the cluster.
__device__ __forceinline__ uint32_t mapa_rank0(uint32_t addr) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(addr));
  return r;
}
// A tile copy into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (cta_group::2).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Accumulator hand-back arrivals (own CTA / CTA 0 of the pair) with relaxed
// semantics. Nothing in memory is published by them: the TMEM loads they
// announce have completed (tcgen05.wait::ld) and are ordered before the
// arrival by tcgen05.fence::before_thread_sync. A release arrival would also
// wait for this thread's earlier writes to become visible, which costs over a
// thousand cycles per tile at cluster scope.
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM allocation; for the pair (cta_group::2) one warp in each of the two CTAs executes it.
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  if constexpr (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 or f16 in, fp32 accumulate).
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// D[tmem of both CTAs] (+)= A[both CTAs' smem] * B[both CTAs' smem]: one M=256 MMA of the pair
// (each CTA holds 128 rows of A, 128 columns of B and its 128 rows of D), issued by CTA 0.
__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at offset `bar` of every CTA in `cta_mask` once the pair's MMAs issued so far are done.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptors (tcgen05 "matrix descriptor" format:
// start address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride
// byte offset >> 4 in 32-45, descriptor version 1 in bits 46-47, swizzle mode
// in 61-63 with 2 = 128-byte swizzle).
//
// A, K-major, 128B swizzle: rows of 128 B (64 elements of K), 8-row groups
// 1024 B apart (stride byte offset); the K extent of one MMA (32 B) lies
// inside the swizzle row, so the leading offset is unused. The k-th K=16 slice
// starts 32*k bytes further.
__device__ __forceinline__ uint64_t desc_a(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}
// B, N-major (MN-major), 128B swizzle: each 64-column box is 64 k-rows of
// 128 B; 8-row k groups are 1024 B apart (stride byte offset) and 64-column
// boxes are B_BOX_BYTES apart (leading byte offset). The k-th K=16 slice (two
// 8-row groups) starts 2048*k bytes further.
__device__ __forceinline__ uint64_t desc_b(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>(B_BOX_BYTES >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// ------------------------------------------------------------ tile decode

struct Tile {
  int job, bb, mt, nt;
};

// Work unit u is a pair of vertically adjacent 128 x 256 tiles with the same
// column block; CTA `rank` of the cluster takes m-tile 2 * pair + rank. Units
// are rasterised in groups of P.group_pairs pairs, column-major inside a group.
__device__ __forceinline__ Tile decode_unit(const TcParams& P, int u, int rank) {
  int lo = 0, hi = P.njobs - 1;
  while (lo < hi) {  // last job with unit_start <= u
    const int mid = (lo + hi + 1) >> 1;
    if (P.unit_start[mid] <= u) lo = mid; else hi = mid - 1;
  }
  const int jm = P.jobs[lo].m, jn = P.jobs[lo].n;
  const int mpairs = (jm + 2 * BM - 1) / (2 * BM), ntiles = (jn + BN - 1) / BN;
  const int local = u - P.unit_start[lo];
  const int per_b = mpairs * ntiles;
  const int GP = P.group_pairs;
  Tile T;
  T.job = lo;
  T.bb = local / per_b;
  const int r = local - T.bb * per_b;
  const int group = r / (GP * ntiles);
  const int first = group * GP;
  const int gp = min(GP, mpairs - first);
  const int in_g = r - group * GP * ntiles;
  T.mt = 2 * (first + in_g % gp) + rank;
  T.nt = in_g / gp;
  return T;
}

// --------------------------------------------------------------- epilogue

__device__ __forceinline__ uint32_t cvt_pair(float a, float b, int out_dtype) {
  if (out_dtype == COCO_F16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Eight 16-bit values (f16 or bf16) of a 16-byte vector as floats.
__device__ __forceinline__ void unpack8(uint4 v, int dtype, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t;
    if (dtype == COCO_F16) t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    else t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Dropout keep test of the FusedAllReduce: element e is kept iff the top 24
// bits of SplitMix64 output number e+1 from state `seed` (Steele, Lea and
// Flood, OOPSLA 2014) are below the threshold; `z` is that output's state,
// seed + (e+1) * gamma. The finaliser's last xor-shift by 31 leaves bits
// 40..63 unchanged, so it is not computed.
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
__device__ __forceinline__ bool keep_state(uint64_t z, uint32_t threshold) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return static_cast<uint32_t>(z >> 40) < threshold;
}

// ------------------------------------------------------------------ kernel

// MODE = EPI_STORE: store the accumulator. MODE = EPI_FUSED_ALLREDUCE: the
// accumulator is a sum over ranks (the K-segments are the ranks' K-slices);
// add the bias, apply dropout and add the residual in registers, then store
// the tile to every replica of the group ([CoCoNet] §5.2, FusedAllReduce,
// with the MatMul of its Fig. 3 fused in front). MODE = EPI_ADD: add the
// output's present values (fp32) to the accumulator and store the sum in
// place ([Decomp] §5.1's Addition fused into the partial einsum, as its §5.4.1
// describes the loop's accumulation).
template <int MODE, bool TWO_SM>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<MODE, TWO_SM>::THREADS, 1)
    k_gemm_tc(const __grid_constant__ TcParams P) {
  using C = Cfg<MODE, TWO_SM>;
  constexpr int STAGES = C::STAGES, EPI_WARPS = C::EPI_WARPS, STAGE_BYTES = C::STAGE;
  constexpr int EPI_OFF = C::EPI_OFF, BAR_OFF = C::BAR_OFF, NUM_BARS = C::NUM_BARS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + BAR_OFF;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + 8 * NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + BAR_OFF + 8 * NUM_BARS + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pair: both CTAs walk the same work units; CTA `rank` takes the unit's m-tile
  // 2 * pair + rank. With one CTA per MMA each CTA loads its A tile and the whole B tile
  // itself; with the pair MMA each loads its A tile and its 128 columns of B.
  const int rank = static_cast<int>(cluster_ctarank());
  const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  constexpr uint16_t kPair = 0x3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      // freed by one commit: the CTA's own MMAs (one CTA per MMA) or CTA 0's pair MMAs
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      // one arrival per epilogue warp; pair MMA: CTA 0's accumulator is free once both CTAs'
      // epilogues have read their halves
      mbar_init(tempty_bar(a), (TWO_SM ? 2 : 1) * EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    if constexpr (MODE != EPI_STORE)
      for (int w = 0; w < EPI_WARPS; ++w) mbar_init(bar0 + 8u * (2 * STAGES + 5 + w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc<TWO_SM>(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  cluster_sync();  // the peer's barriers exist before the pair MMA's copies or commits reach them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicCAS(P.err, 0u, static_cast<unsigned int>(COCO_ERR_TIMEOUT));
  };

  // The MMA role is run by a whole warp so that every loop value is
  // warp-uniform; one elected lane issues the MMAs. Run by a single lane, the
  // same loop keeps its values in per-thread registers and no longer keeps the
  // tensor pipe fed. The producer is run the same way for the pair MMA, whose
  // long, operand-bound k-loops gain from it (the K=512 MatMul: 10 % faster);
  // with one CTA per MMA (short k-loops whose tiles are store-bound, like the
  // K=128 batched einsum) a single-lane producer measured 10 % faster.
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    // (lanes 1..31 of a single-lane producer go straight to the final barrier)
    if (TWO_SM || lane == 0) {
      const bool leader = TWO_SM ? elect_one() : true;
      auto wait = [&](uint32_t bar, uint32_t parity, volatile int* flag) {
        if constexpr (TWO_SM) return mbar_wait_warp(bar, parity, flag);
        else return mbar_wait(bar, parity, flag);
      };
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per stage: a copy was issued, and the phase it completes
      bool ok = true;
      // Producers in step: with wave_sync, wave i of the grid (every cluster's i-th unit) starts
      // loading only when every producer has issued wave i-1, so the pairs of a wave stream the same
      // operand slices at the same time and L2 serves them once (the large-B, long-K case: 3% faster
      // there, at a higher clock for the DRAM power saved). The wait is bounded like every other.
      const int full_waves = P.total_units / nclusters;
      int iu = 0;
      for (int u = cluster_id; ok && u < P.total_units; u += nclusters, ++iu) {
        if (P.wave_sync && iu >= 1 && iu < full_waves) {
          bool synced = true;
          if (leader) {
            atomicAdd(P.wave_counter, 1u);
            const unsigned int want = static_cast<unsigned int>(iu) * gridDim.x;
            const uint64_t t0 = globaltimer();
            while (atomicAdd(P.wave_counter, 0u) < want) {
              if (*abort_flag || globaltimer() - t0 > kTimeoutNs) {
                synced = false;
                break;
              }
              __nanosleep(64);
            }
          }
          if constexpr (TWO_SM) synced = __shfl_sync(0xffffffffu, synced ? 1 : 0, 0) != 0;
          if (!synced) {
            if (leader) fail();
            ok = false;
            break;
          }
        }
        const Tile T = decode_unit(P, u, rank);
        const Job J = P.jobs[T.job];  // a register copy: asm memory clobbers would force reloads
        for (int si = 0; ok && si < J.nseg; ++si) {
          const Seg S = P.segs[J.seg0 + si];
          const CUtensorMap* ma = &P.maps[S.a];
          const CUtensorMap* mb = &P.maps[S.b];
          const int kblocks = (S.klen + BK - 1) / BK;
          const int arow = S.a_r0 + T.mt * BM, ab = S.a_b0 + T.bb;
          const int bcol = S.b_c0 + T.nt * BN, bb = S.b_b0 + T.bb;
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
              if (leader) fail();
              ok = false;
              break;
            }
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
            if (leader) {
              if constexpr (TWO_SM) {
                // both CTAs' copies complete CTA 0's barrier, which expects the pair's bytes
                const uint32_t fb = mapa_rank0(full_bar(stage));
                if (rank == 0) mbar_expect_tx(full_bar(stage), 2 * STAGE_BYTES);
                tma_load_3d_pair(sa, ma, fb, S.a_k0 + kb * BK, arow, ab);
#pragma unroll
                for (int j = 0; j < BN / 128; ++j)  // this CTA's 128 columns of B
                  tma_load_3d_pair(sb + j * B_BOX_BYTES, mb, fb, bcol + rank * (BN / 2) + 64 * j, S.b_k0 + kb * BK,
                                   bb);
              } else {
                mbar_expect_tx(full_bar(stage), STAGE_BYTES);  // own A + the whole B tile
                tma_load_3d(sa, ma, full_bar(stage), S.a_k0 + kb * BK, arow, ab);
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                  tma_load_3d(sb + j * B_BOX_BYTES, mb, full_bar(stage), bcol + 64 * j, S.b_k0 + kb * BK, bb);
              }
            }
            if constexpr (TWO_SM) __syncwarp();
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
      if (!ok && (!TWO_SM || rank == 0)) {  // let copies in flight land (pair: CTA 0's barriers count both)
        int dummy = 0;
        volatile int* never = &dummy;
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u) wait(full_bar(s), (issued_parity >> s) & 1u, never);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (!TWO_SM || rank == 0) {  // pair MMA: CTA 0 issues for both
      // The tensor pipe finishes a k-block (four K=16 MMAs) in about 512
      // cycles, so per-k-block work stays at a few instructions: descriptors
      // advance by adding to the encoded start address (stage offsets stay
      // below the 14-bit field's limit, as shared memory ends below 256 KB),
      // the job is followed by a forward scan (units increase monotonically),
      // and only the k-block count is read per tile. tcgen05.commit tracks the
      // MMAs of the thread that issues it, so one lane issues both.
      const bool leader = elect_one();
      const uint32_t idesc = P.idesc;
      const uint64_t adesc0 = desc_a(sbase), bdesc0 = desc_b(sbase + A_BYTES);
      constexpr uint32_t kStageDesc = static_cast<uint32_t>(STAGE_BYTES >> 4);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      int job = 0;
      bool ok = true;
      bool any_mma = false;
      for (int u = cluster_id; ok && u < P.total_units; u += nclusters, ++local) {
        while (job + 1 < P.njobs && P.unit_start[job + 1] <= u) ++job;
        const int kblocks = P.jobs[job].kblocks;
        const int acc = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!mbar_wait_warp(tempty_bar(acc), aph ^ 1u, abort_flag)) {
          if (leader) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_warp(full_bar(stage), phase, abort_flag)) {
            if (leader) fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t off = static_cast<uint64_t>(stage * kStageDesc);
          const uint64_t ad = adesc0 + off, bd = bdesc0 + off;
          if (leader) {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              // K-major A: the k-th K=16 slice is 32 B further; N-major B: 2048 B (in 16-byte units)
              const uint32_t accumulate = (kb | k) != 0;
              if constexpr (TWO_SM) umma_pair(d, ad + 2 * k, bd + 128 * k, idesc, accumulate);
              else umma(d, ad + 2 * k, bd + 128 * k, idesc, accumulate);
            }
            // the stage may be refilled (pair MMA: by both CTAs' producers)
            if constexpr (TWO_SM) umma_commit_pair(empty_bar(stage), kPair);
            else umma_commit(empty_bar(stage));
          }
          __syncwarp();
          any_mma = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok && leader) {
          if constexpr (TWO_SM) umma_commit_pair(tfull_bar(acc), kPair);  // both epilogues may read their halves
          else umma_commit(tfull_bar(acc));
        }
        __syncwarp();
      }
      if (!ok && any_mma) {  // wait for the MMAs already issued before TMEM is freed
        if (leader) {
          if constexpr (TWO_SM) umma_commit_pair(drain_bar, 0x1);
          else umma_commit(drain_bar);
        }
        __syncwarp();
        int dummy = 0;
        volatile int* never = &dummy;
        mbar_wait_warp(drain_bar, 0, never);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
    const uint32_t strips = sbase + EPI_OFF + (warp - 2) * C::STRIPS * EPI_STRIP;
    const uint32_t res_strip = strips + EPI_STRIP;  // fused mode only
    const uint32_t res_bar = bar0 + 8u * (2 * STAGES + 5 + (warp - 2));
    uint32_t res_phase = 0;
    bool res_pending = false;
    // with 8 epilogue warps, warps 2..5 take columns [0, BN/2) and warps 6..9 [BN/2, BN)
    constexpr int COLS = EPI_WARPS == 8 ? BN / 2 : BN;
    const int col_begin = EPI_WARPS == 8 ? ((warp - 2) >> 2) * COLS : 0;
    const uint64_t seed = P.seed;
    const uint32_t keep_threshold = P.keep_threshold;
    const float scale = P.scale;
    const bool dropout = P.dropout != 0;
    const char* bias_ptr = static_cast<const char*>(P.bias);
    uint64_t evict_first = 0;  // L2 policy for data touched once (outputs, residual)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
    const int out_dt = P.out_dtype;
    const int esize = out_dt == COCO_F32 ? 4 : 2;
    const int cols_per_chunk = 128 / esize;  // 32 (fp32) or 64 (16-bit): one 128-byte strip row
    const int vec_elems = 16 / esize;
    int local = 0;
    int buf = 0;
    for (int u = cluster_id; u < P.total_units; u += nclusters, ++local) {
      const Tile T = decode_unit(P, u, rank);
      const Job J = P.jobs[T.job];  // a register copy: asm memory clobbers would force reloads
      const OutView O = P.outs[J.out];
      const int acc = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      const int row0 = T.mt * BM + quarter * 32;  // job-relative row of this warp's lane 0
      const bool has_res = MODE != EPI_STORE && J.res != nullptr;
      auto load_residual = [&](int cc) {  // lane 0 only
        mbar_expect_tx(res_bar, EPI_STRIP);
        tma_load_3d(res_strip, &P.omaps[J.res_map], res_bar, J.o_c0 + T.nt * BN + cc, J.o_r0 + row0,
                    J.o_b0 + T.bb);
      };
      // Operands of the FusedAllReduce epilogue that do not depend on the
      // accumulator are requested before it is ready: the first residual strip
      // (the strip is free: the previous tile's last chunk issued no load), and
      // the bias, lane l holding tile columns [8l, 8l + 8) for the lanes that
      // need them (shuffles), instead of one dependent global load per column group.
      uint4 bias_v = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (MODE != EPI_STORE) {
        if (has_res && lane == 0) {
          load_residual(col_begin);
          res_pending = true;
        }
      }
      if constexpr (MODE == EPI_FUSED_ALLREDUCE) {
        const int bc = J.o_c0 + T.nt * BN + 8 * lane;
        if (bias_ptr && bc < O.cols) bias_v = ld_nc_v4(bias_ptr + bc * 2);
      }
      // all lanes must agree before the warp-collective TMEM loads
      const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, abort_flag));
      if (!ready) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      // A bulk store clips only at the tensor's edges, so it is used when the
      // tile lies inside its job's region or overhangs only past the tensor.
      const bool bulk = (T.mt * BM + BM <= J.m || J.o_r0 + J.m == O.rows) &&
                        (T.nt * BN + BN <= J.n || J.o_c0 + J.n == O.cols);
      const int64_t obatch = static_cast<int64_t>(J.o_b0 + T.bb) * O.bstride;
      const int jrow = row0 + lane;
      const int64_t grow = J.o_r0 + jrow;
      for (int c0 = col_begin; c0 < col_begin + COLS; c0 += cols_per_chunk) {
        const bool last = c0 + cols_per_chunk >= col_begin + COLS;
        uint32_t p[32];
        if constexpr (MODE == EPI_ADD) {
          // fp32 output: 32 columns of this lane's row, plus the same columns of the output as they were
          // (the addend strip, loaded by TMA one chunk ahead)
          uint4 cur[8];
          const bool landed = __all_sync(0xffffffffu, mbar_wait(res_bar, res_phase, abort_flag));
          if (!landed) {
            if (lane == 0) fail();
            break;
          }
          res_phase ^= 1u;
#pragma unroll
          for (int c = 0; c < 8; ++c) cur[c] = ld_shared_v4(res_strip + lane * 128 + ((c ^ (lane & 7)) << 4));
          fence_proxy_async_smem();  // these reads come before the next TMA write of the strip
          __syncwarp();
          if (lane == 0) {
            res_pending = !last;
            if (!last) load_residual(c0 + cols_per_chunk);
          }
          uint32_t r[32];
          tmem_ld32(tbase + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            p[4 * c + 0] = __float_as_uint(__uint_as_float(cur[c].x) + __uint_as_float(r[4 * c + 0]));
            p[4 * c + 1] = __float_as_uint(__uint_as_float(cur[c].y) + __uint_as_float(r[4 * c + 1]));
            p[4 * c + 2] = __float_as_uint(__uint_as_float(cur[c].z) + __uint_as_float(r[4 * c + 2]));
            p[4 * c + 3] = __float_as_uint(__uint_as_float(cur[c].w) + __uint_as_float(r[4 * c + 3]));
          }
        } else if constexpr (MODE == EPI_FUSED_ALLREDUCE) {
          // 16-bit output: 64 columns of this lane's row
          const int gcol0 = J.o_c0 + T.nt * BN + c0;
          uint4 cur[8];
          if (has_res) {
            const bool landed = __all_sync(0xffffffffu, mbar_wait(res_bar, res_phase, abort_flag));
            if (!landed) {
              if (lane == 0) fail();
              break;
            }
            res_phase ^= 1u;
#pragma unroll
            for (int c = 0; c < 8; ++c) cur[c] = ld_shared_v4(res_strip + lane * 128 + ((c ^ (lane & 7)) << 4));
            fence_proxy_async_smem();  // these reads come before the next TMA write of the strip
            __syncwarp();
            if (lane == 0) {
              res_pending = !last;
              if (!last) load_residual(c0 + cols_per_chunk);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) cur[c] = make_uint4(0u, 0u, 0u, 0u);
          }
          uint32_t r[32], r2[32];
          tmem_ld32(tbase + c0, r);
          tmem_ld32(tbase + c0 + 32, r2);
          tmem_ld_wait();
          uint64_t z = seed + (static_cast<uint64_t>(grow * O.cols + gcol0) + 1ull) * kGamma;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float bias[8], res[8], v[8];
            const int src = (c0 >> 3) + i;  // the lane holding tile columns c0 + 8i .. + 7
            uint4 bv;
            bv.x = __shfl_sync(0xffffffffu, bias_v.x, src);
            bv.y = __shfl_sync(0xffffffffu, bias_v.y, src);
            bv.z = __shfl_sync(0xffffffffu, bias_v.z, src);
            bv.w = __shfl_sync(0xffffffffu, bias_v.w, src);
            unpack8(bv, out_dt, bias);
            unpack8(cur[i], out_dt, res);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int c = i * 8 + j;
              float x = __uint_as_float(c < 32 ? r[c] : r2[c - 32]) + bias[j];
              if (dropout) x = keep_state(z, keep_threshold) ? x * scale : 0.0f;
              v[j] = x + res[j];
              z += kGamma;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) p[i * 4 + j] = cvt_pair(v[2 * j], v[2 * j + 1], out_dt);
          }
        } else if (out_dt == COCO_F32) {
          tmem_ld32(tbase + c0, p);
          tmem_ld_wait();
        } else {
          uint32_t r[32], r2[32];
          tmem_ld32(tbase + c0, r);
          tmem_ld32(tbase + c0 + 32, r2);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            p[i] = cvt_pair(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), out_dt);
            p[16 + i] = cvt_pair(__uint_as_float(r2[2 * i]), __uint_as_float(r2[2 * i + 1]), out_dt);
          }
        }
        if (last) {  // the accumulator is in registers: hand TMEM back to the MMA warp now
          tc_fence_before();
          __syncwarp();  // every lane's TMEM loads are complete before one lane releases for the warp
          if (lane == 0) {
            if constexpr (TWO_SM) mbar_arrive_cluster_relaxed(mapa_rank0(tempty_bar(acc)));
            else mbar_arrive_relaxed(tempty_bar(acc));
          }
        }
        // the strip about to be overwritten was handed to a bulk store two chunks ago (FusedAllReduce:
        // its one output strip, to the stores of the previous chunk). Chunks stored with plain stores
        // commit no bulk group, so after a bulk-stored tile the group count no longer tells which
        // strip is free: such chunks wait for every earlier bulk store to have read its strip.
        if (lane == 0) {
          if (MODE != EPI_STORE || !bulk) bulk_wait_read_all();
          else bulk_wait_read_le1();
        }
        __syncwarp();
        const uint32_t strip = MODE != EPI_STORE ? strips : strips + buf * EPI_STRIP;
#pragma unroll
        for (int c = 0; c < 8; ++c)  // row = lane, 16-byte chunk c at its 128-byte-swizzle slot
          st_shared_v4(strip + lane * 128 + ((c ^ (lane & 7)) << 4), p[4 * c], p[4 * c + 1], p[4 * c + 2],
                       p[4 * c + 3]);
        if (bulk) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {  // one strip, stored to every replica of the job's output
            const int nrep = MODE == EPI_STORE ? 1 : J.nout;
            for (int o = 0; o < nrep; ++o)
              tma_store_3d(&P.omaps[J.out + o], strip, J.o_c0 + T.nt * BN + c0, J.o_r0 + row0, J.o_b0 + T.bb,
                           evict_first);
            bulk_commit();
          }
        } else {
          __syncwarp();
          // strip -> global: 8 lanes per 128-byte row segment, 4 rows per pass, bounded by the job
          const int ch = lane & 7;
          const int col = T.nt * BN + c0 + ch * vec_elems;  // job-relative column
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int rr = it * 4 + (lane >> 3);
            const int row = row0 + rr;
            const uint4 v = ld_shared_v4(strip + rr * 128 + ((ch ^ (rr & 7)) << 4));
            if (row < J.m && col < J.n) {
              const int64_t off = obatch + static_cast<int64_t>(J.o_r0 + row) * O.ld + (J.o_c0 + col);
              if (MODE == EPI_STORE) {
                *reinterpret_cast<uint4*>(static_cast<char*>(O.ptr) + off * esize) = v;
              } else {
                for (int o = 0; o < J.nout; ++o)
                  *reinterpret_cast<uint4*>(static_cast<char*>(P.outs[J.out + o].ptr) + off * esize) = v;
              }
            }
          }
          __syncwarp();
        }
        buf ^= 1;
      }
    }
    if (lane == 0) {
      if (res_pending) {  // an aborted tile may leave a residual load in flight
        int dummy = 0;
        volatile int* never = &dummy;
        mbar_wait(res_bar, res_phase, never);
      }
      bulk_wait_all();  // bulk stores finish before the CTA's shared memory goes away
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers or read its TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<TWO_SM>(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------ B-stationary short-K kernel
//
// Jobs that contract over at most BS_KB k-blocks (K <= 128, such as the
// batched einsum of [Decomp] §5.1 case 3) are bound by their output stream: a
// 128 x 256 tile's MMAs take about a quarter of the time its bf16 results
// take to reach HBM. In k_gemm_tc each such tile also loads a 32 KB A tile
// and a 64 KB B tile through the SM's TMA unit, which the stores share. Here
// a CTA keeps one B tile [K x 256] in shared memory for a unit of up to
// BS_MTILES vertically adjacent m-tiles and streams only their A tiles:
// 48 KB of operand loads per output tile instead of 96 KB.
//
// One CTA per SM, no cluster. Warp 0 (one lane) loads B once per unit (two B
// buffers, so the next unit's B arrives while this unit's MMAs run) and A
// once per tile, warp 1 issues one M=128, N=256 MMA per K=16 step from an
// elected lane into one of two TMEM accumulators, warps 2..5 store as in
// k_gemm_tc (a ring of BS_STRIPS strips per warp). Units are numbered with
// the n-tile innermost, so CTAs running side by side read the same A tiles,
// and the two m-halves of a B tile are BS_MTILES units apart.
constexpr int BS_KB = 2;
constexpr int BS_MTILES = 4;
constexpr int BS_B_BUFS = 2;
constexpr int BS_A_STAGES = 2;
constexpr int BS_STRIPS = 2;
constexpr int BS_EPI_WARPS = 4;  // one per TMEM lane quarter (8, two per quarter, measured 6 % slower)
constexpr int BS_B_TILE = BS_KB * B_BYTES;  // 64 KB
constexpr int BS_A_TILE = BS_KB * A_BYTES;  // 32 KB
struct BsCfg {
  static constexpr int EPI_WARPS = BS_EPI_WARPS;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int A_OFF = BS_B_BUFS * BS_B_TILE;
  static constexpr int EPI_OFF = A_OFF + BS_A_STAGES * BS_A_TILE;
  static constexpr int BAR_OFF = EPI_OFF + EPI_WARPS * BS_STRIPS * EPI_STRIP;
  // B full x bufs, B empty x bufs, A full x stages, A empty x stages, TMEM full x2, TMEM empty x2, drain
  static constexpr int NUM_BARS = 2 * BS_B_BUFS + 2 * BS_A_STAGES + 5;
  static constexpr int SMEM_BYTES = BAR_OFF + 8 * NUM_BARS + 16 + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
};

// At most N committed bulk groups may still be reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read_le() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

struct BsUnit {
  int job, bb, mt0, ntm, nt;
};

// Unit u of a B-stationary launch: (job, batch, m-chunk, n-tile), n-tile innermost.
__device__ __forceinline__ BsUnit bs_decode(const TcParams& P, int u) {
  int lo = 0, hi = P.njobs - 1;
  while (lo < hi) {  // last job with unit_start <= u
    const int mid = (lo + hi + 1) >> 1;
    if (P.unit_start[mid] <= u) lo = mid; else hi = mid - 1;
  }
  const int mtiles = (P.jobs[lo].m + BM - 1) / BM, ntiles = (P.jobs[lo].n + BN - 1) / BN;
  const int mch = (mtiles + BS_MTILES - 1) / BS_MTILES;
  const int local = u - P.unit_start[lo];
  const int per_b = mch * ntiles;
  BsUnit U;
  U.job = lo;
  U.bb = local / per_b;
  const int r = local - U.bb * per_b;
  const int mc = r / ntiles;
  U.nt = r - mc * ntiles;
  U.mt0 = mc * BS_MTILES;
  U.ntm = min(BS_MTILES, mtiles - U.mt0);
  return U;
}

__global__ void __launch_bounds__(BsCfg::THREADS, 1) k_gemm_tc_bs(const __grid_constant__ TcParams P) {
  constexpr int A_OFF = BsCfg::A_OFF, EPI_OFF = BsCfg::EPI_OFF, BAR_OFF = BsCfg::BAR_OFF;
  constexpr int NUM_BARS = BsCfg::NUM_BARS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + BAR_OFF;
  constexpr uint32_t ABAR = 16u * BS_B_BUFS;  // offset of the A barriers
  auto bfull = [&](int b) { return bar0 + 8u * b; };
  auto bempty = [&](int b) { return bar0 + 8u * (BS_B_BUFS + b); };
  auto afull = [&](int s) { return bar0 + ABAR + 8u * s; };
  auto aempty = [&](int s) { return bar0 + ABAR + 8u * (BS_A_STAGES + s); };
  auto tfull = [&](int a) { return bar0 + ABAR + 8u * (2 * BS_A_STAGES + a); };
  auto tempty = [&](int a) { return bar0 + ABAR + 8u * (2 * BS_A_STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + ABAR + 8u * (2 * BS_A_STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + 8 * NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + BAR_OFF + 8 * NUM_BARS + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < BS_B_BUFS; ++b) {
      mbar_init(bfull(b), 1);
      mbar_init(bempty(b), 1);
    }
    for (int s = 0; s < BS_A_STAGES; ++s) {
      mbar_init(afull(s), 1);
      mbar_init(aempty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), BsCfg::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc<false>(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicCAS(P.err, 0u, static_cast<unsigned int>(COCO_ERR_TIMEOUT));
  };

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer (lane 0)
    if (lane == 0) {
      int bb_ = 0;  // B buffer of the next unit
      uint32_t bphase = 0;
      uint32_t b_issued = 0, b_parity = 0;  // per B buffer: a copy was issued, and the phase it completes
      int st = 0;
      uint32_t aph = 0;
      uint32_t issued = 0, issued_parity = 0;  // per A stage: a copy was issued, and the phase it completes
      bool ok = true;
      for (int u = blockIdx.x; ok && u < P.total_units; u += gridDim.x) {
        const BsUnit U = bs_decode(P, u);
        const Job J = P.jobs[U.job];
        // the unit's B tile: every k-block of every segment, in segment order
        if (!mbar_wait(bempty(bb_), bphase ^ 1u, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        mbar_expect_tx(bfull(bb_), static_cast<uint32_t>(J.kblocks * B_BYTES));
        {
          const uint32_t sbt = sbase + bb_ * BS_B_TILE;
          int kb = 0;
          for (int si = 0; si < J.nseg; ++si) {
            const Seg S = P.segs[J.seg0 + si];
            const int kbs = (S.klen + BK - 1) / BK;
            for (int k = 0; k < kbs; ++k, ++kb)
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_3d(sbt + kb * B_BYTES + j * B_BOX_BYTES, &P.maps[S.b], bfull(bb_),
                            S.b_c0 + U.nt * BN + 64 * j, S.b_k0 + k * BK, S.b_b0 + U.bb);
          }
        }
        b_issued |= 1u << bb_;
        b_parity = (b_parity & ~(1u << bb_)) | (bphase << bb_);
        if (++bb_ == BS_B_BUFS) { bb_ = 0; bphase ^= 1u; }
        // its m-tiles' A tiles
        for (int t = 0; t < U.ntm; ++t) {
          if (!mbar_wait(aempty(st), aph ^ 1u, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t sa = sbase + A_OFF + st * BS_A_TILE;
          mbar_expect_tx(afull(st), static_cast<uint32_t>(J.kblocks * A_BYTES));
          int kb = 0;
          for (int si = 0; si < J.nseg; ++si) {
            const Seg S = P.segs[J.seg0 + si];
            const int kbs = (S.klen + BK - 1) / BK;
            for (int k = 0; k < kbs; ++k, ++kb)
              tma_load_3d(sa + kb * A_BYTES, &P.maps[S.a], afull(st), S.a_k0 + k * BK,
                          S.a_r0 + (U.mt0 + t) * BM, S.a_b0 + U.bb);
          }
          issued |= 1u << st;
          issued_parity = (issued_parity & ~(1u << st)) | (aph << st);
          if (++st == BS_A_STAGES) { st = 0; aph ^= 1u; }
        }
      }
      if (!ok) {  // let copies in flight land before the CTA's shared memory goes away
        int dummy = 0;
        volatile int* never = &dummy;
        for (int b = 0; b < BS_B_BUFS; ++b)
          if ((b_issued >> b) & 1u) mbar_wait(bfull(b), (b_parity >> b) & 1u, never);
        for (int s = 0; s < BS_A_STAGES; ++s)
          if ((issued >> s) & 1u) mbar_wait(afull(s), (issued_parity >> s) & 1u, never);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    const uint32_t idesc = P.idesc;
    int bb_ = 0;
    uint32_t bphase = 0;
    int st = 0;
    uint32_t aph = 0;
    int lt = 0;  // tiles of this CTA so far
    bool ok = true, any_mma = false;
    for (int u = blockIdx.x; ok && u < P.total_units; u += gridDim.x) {
      const BsUnit U = bs_decode(P, u);
      const int kblocks = P.jobs[U.job].kblocks;
      if (!mbar_wait_warp(bfull(bb_), bphase, abort_flag)) {
        if (leader) fail();
        ok = false;
        break;
      }
      const uint32_t sbt = sbase + bb_ * BS_B_TILE;
      tc_fence_after();
      for (int t = 0; t < U.ntm; ++t, ++lt) {
        const int acc = lt & 1;
        const uint32_t tph = (lt >> 1) & 1;
        if (!mbar_wait_warp(tempty(acc), tph ^ 1u, abort_flag) || !mbar_wait_warp(afull(st), aph, abort_flag)) {
          if (leader) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        if (leader) {
          for (int kb = 0; kb < kblocks; ++kb) {
            const uint64_t ad = desc_a(sbase + A_OFF + st * BS_A_TILE + kb * A_BYTES);
            const uint64_t bd = desc_b(sbt + kb * B_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) umma(d, ad + 2 * k, bd + 128 * k, idesc, (kb | k) != 0);
          }
          umma_commit(aempty(st));  // the A stage may be refilled
          umma_commit(tfull(acc));  // the epilogue may read the accumulator
        }
        __syncwarp();
        any_mma = true;
        if (++st == BS_A_STAGES) { st = 0; aph ^= 1u; }
      }
      if (ok && leader) umma_commit(bempty(bb_));  // the unit's B buffer may be refilled
      __syncwarp();
      if (++bb_ == BS_B_BUFS) { bb_ = 0; bphase ^= 1u; }
    }
    if (!ok && any_mma) {  // wait for the MMAs already issued before TMEM is freed
      if (leader) umma_commit(drain_bar);
      __syncwarp();
      int dummy = 0;
      volatile int* never = &dummy;
      mbar_wait_warp(drain_bar, 0, never);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
    const uint32_t strips = sbase + EPI_OFF + (warp - 2) * BS_STRIPS * EPI_STRIP;
    constexpr int COLS = BN / (BsCfg::EPI_WARPS / 4);  // columns of a tile this warp stores
    const int col_begin = ((warp - 2) >> 2) * COLS;
    uint64_t evict_first = 0;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
    const int out_dt = P.out_dtype;
    const int esize = out_dt == COCO_F32 ? 4 : 2;
    const int cols_per_chunk = 128 / esize;
    const int vec_elems = 16 / esize;
    int lt = 0, buf = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < P.total_units; u += gridDim.x) {
      const BsUnit U = bs_decode(P, u);
      const Job J = P.jobs[U.job];
      const OutView O = P.outs[J.out];
      const int64_t obatch = static_cast<int64_t>(J.o_b0 + U.bb) * O.bstride;
      for (int t = 0; t < U.ntm; ++t, ++lt) {
        const int mt = U.mt0 + t;
        const int acc = lt & 1;
        const uint32_t tph = (lt >> 1) & 1;
        const int row0 = mt * BM + quarter * 32;  // job-relative row of this warp's lane 0
        const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull(acc), tph, abort_flag));
        if (!ready) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
        const bool bulk = (mt * BM + BM <= J.m || J.o_r0 + J.m == O.rows) &&
                          (U.nt * BN + BN <= J.n || J.o_c0 + J.n == O.cols);
        for (int c0 = col_begin; c0 < col_begin + COLS; c0 += cols_per_chunk) {
          const bool last = c0 + cols_per_chunk >= col_begin + COLS;
          uint32_t p[32];
          if (out_dt == COCO_F32) {
            tmem_ld32(tbase + c0, p);
            tmem_ld_wait();
          } else {
            uint32_t r[32], r2[32];
            tmem_ld32(tbase + c0, r);
            tmem_ld32(tbase + c0 + 32, r2);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              p[i] = cvt_pair(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), out_dt);
              p[16 + i] = cvt_pair(__uint_as_float(r2[2 * i]), __uint_as_float(r2[2 * i + 1]), out_dt);
            }
          }
          if (last) {  // this warp's part of the accumulator is in registers: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(tempty(acc));
          }
          // the strip about to be overwritten was handed to a bulk store BS_STRIPS chunks ago; chunks
          // stored with plain stores commit no group, so they wait for every earlier bulk store
          if (lane == 0) {
            if (bulk) bulk_wait_read_le<BS_STRIPS - 1>();
            else bulk_wait_read_all();
          }
          __syncwarp();
          const uint32_t strip = strips + buf * EPI_STRIP;
#pragma unroll
          for (int c = 0; c < 8; ++c)  // row = lane, 16-byte chunk c at its 128-byte-swizzle slot
            st_shared_v4(strip + lane * 128 + ((c ^ (lane & 7)) << 4), p[4 * c], p[4 * c + 1], p[4 * c + 2],
                         p[4 * c + 3]);
          if (bulk) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&P.omaps[J.out], strip, J.o_c0 + U.nt * BN + c0, J.o_r0 + row0, J.o_b0 + U.bb,
                           evict_first);
              bulk_commit();
            }
          } else {
            __syncwarp();
            // strip -> global: 8 lanes per 128-byte row segment, 4 rows per pass, bounded by the job
            const int ch = lane & 7;
            const int col = U.nt * BN + c0 + ch * vec_elems;  // job-relative column
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int rr = it * 4 + (lane >> 3);
              const int row = row0 + rr;
              const uint4 v = ld_shared_v4(strip + rr * 128 + ((ch ^ (rr & 7)) << 4));
              if (row < J.m && col < J.n) {
                const int64_t off = obatch + static_cast<int64_t>(J.o_r0 + row) * O.ld + (J.o_c0 + col);
                *reinterpret_cast<uint4*>(static_cast<char*>(O.ptr) + off * esize) = v;
              }
            }
            __syncwarp();
          }
          if (++buf == BS_STRIPS) buf = 0;
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // bulk stores finish before the CTA's shared memory goes away
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<false>(tmem_base, TMEM_COLS);
  }
}

// Failure-path self-test: the TMEM owner allocates, a consumer warp waits for a
// phase that nothing completes, with the same bounded wait as the GEMM's roles
// but a caller-chosen limit; on expiry it records COCO_ERR_TIMEOUT and raises
// the abort flag, and the owner frees TMEM before every thread returns.
__global__ void __launch_bounds__(64, 1) k_wait_selftest(unsigned int* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc<false>(smem_u32(&tslot), 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  if (warp == 1) {
    const bool ok = mbar_wait_warp(smem_u32(&bar), 0, abort_flag, timeout_ns);
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicCAS(err, 0u, static_cast<unsigned int>(COCO_ERR_TIMEOUT));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<false>(tmem, 32);
  }
}

// ------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A operand: [nb][rows][cols=K], box {64 k, 128 rows}. B operand: [nb][rows=K][cols=N], box {64 n, 64 k}.
bool encode_view(CUtensorMap* map, const View& v, int dtype, bool is_a) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int es = 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(v.cols), static_cast<cuuint64_t>(v.rows),
                        static_cast<cuuint64_t>(v.nb)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(v.ld) * es, static_cast<cuuint64_t>(v.bstride) * es};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(is_a ? BM : BK), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == COCO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, dt, 3, const_cast<void*>(v.ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output map: [nb][rows][cols] of the output dtype, box {128 bytes of columns, 32 rows, 1}, 128B swizzle.
bool encode_out(CUtensorMap* map, const OutView& o, int dtype) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int es = dtype == COCO_F32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(o.cols), static_cast<cuuint64_t>(o.rows),
                        static_cast<cuuint64_t>(o.nb)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(o.ld) * es, static_cast<cuuint64_t>(o.bstride) * es};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = dtype == COCO_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == COCO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, dt, 3, o.ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// per kernel variant and device: the dynamic shared-memory limit was raised (static storage: starts false;
// atomic because calls may come from several host threads, which at worst both set the attribute)
std::atomic<bool> smem_configured[7][64];

}  // namespace

static __device__ unsigned int g_gemm_error = 0;
// Arrival counters of wave-synchronised launches; a launch takes the next slot (launches in flight at
// once must number fewer than the slots).
constexpr int kWaveSlots = 1024;
static __device__ unsigned int g_wave_counters[kWaveSlots];
static std::atomic<unsigned int> g_wave_slot{0};

unsigned int* gemm_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_gemm_error) != cudaSuccess) return nullptr;
  return static_cast<unsigned int*>(p);
}

// Splits the plan into launches that fit the parameter block, remapping view,
// segment and output indices, then launches each.
// Plans are turned into launches in two steps: tc_prepare encodes every
// tensor map and fills the parameter blocks (host work only, no stream
// operation), tc_launch enqueues them. A prepared plan may be launched any
// number of times; only the error word and the arrival counter of a
// cooperative launch are set per launch.
struct TcPrepared {
  void (*kernel)(TcParams) = nullptr;
  int smem = 0, threads = 0;
  std::vector<std::unique_ptr<TcParams>> params;  // one per launch (wave_sync: the launch wants it)
  std::vector<int> grids;
};

void tc_free(TcPrepared* p) { delete p; }

cudaError_t tc_prepare(const GemmPlan& plan, TcPrepared** out) {
  *out = nullptr;
  if (!encode_fn()) return cudaErrorNotSupported;
  const bool far = plan.mode == EPI_FUSED_ALLREDUCE;
  const bool add = plan.mode == EPI_ADD;
  if (far && plan.out_dtype == COCO_F32) return cudaErrorNotSupported;
  if (add && plan.out_dtype != COCO_F32) return cudaErrorNotSupported;
  // Every job (one output region's whole K-segment loop) must fit one launch's parameter block:
  // checked for all jobs before anything is launched, so an unsupported plan runs nothing.
  for (const Job& J : plan.jobs) {
    std::vector<int> as, bs;
    for (int k = 0; k < J.nseg; ++k) {
      const Seg& S = plan.segs[J.seg0 + k];
      if (std::find(as.begin(), as.end(), S.a) == as.end()) as.push_back(S.a);
      if (std::find(bs.begin(), bs.end(), S.b) == bs.end()) bs.push_back(S.b);
    }
    if (static_cast<int>(as.size() + bs.size()) > MAX_MAPS || J.nseg > MAX_SEGS ||
        J.nout + ((far || add) && J.res ? 1 : 0) > MAX_OUTS)
      return cudaErrorNotSupported;
  }
  // k-blocks per tile, averaged over the plan's jobs
  int64_t kb_sum = 0;
  for (const Job& J : plan.jobs)
    for (int k = 0; k < J.nseg; ++k) kb_sum += (plan.segs[J.seg0 + k].klen + BK - 1) / BK;
  const bool two_sm = plan.jobs.empty() ? true : kb_sum >= static_cast<int64_t>(kTwoSmMinKBlocks) * plan.jobs.size();
  // jobs of at most BS_KB k-blocks are store-bound: the B-stationary kernel halves their operand loads
  bool bs = plan.mode == EPI_STORE && !plan.jobs.empty();
  for (const Job& J : plan.jobs) {
    int kb = 0;
    for (int k = 0; k < J.nseg; ++k) kb += (plan.segs[J.seg0 + k].klen + BK - 1) / BK;
    bs = bs && kb <= BS_KB;
  }
  const int variant = bs ? 4 : (add ? 5 : far ? 2 : 0) + (two_sm ? 1 : 0);
  void (*kernel)(TcParams) = nullptr;
  int smem = 0, threads = 0;
  switch (variant) {
    case 4: kernel = k_gemm_tc_bs; smem = BsCfg::SMEM_BYTES; threads = BsCfg::THREADS; break;
    case 0: kernel = k_gemm_tc<EPI_STORE, false>; smem = Cfg<EPI_STORE, false>::SMEM_BYTES;
            threads = Cfg<EPI_STORE, false>::THREADS; break;
    case 1: kernel = k_gemm_tc<EPI_STORE, true>; smem = Cfg<EPI_STORE, true>::SMEM_BYTES;
            threads = Cfg<EPI_STORE, true>::THREADS; break;
    case 2: kernel = k_gemm_tc<EPI_FUSED_ALLREDUCE, false>; smem = Cfg<EPI_FUSED_ALLREDUCE, false>::SMEM_BYTES;
            threads = Cfg<EPI_FUSED_ALLREDUCE, false>::THREADS; break;
    case 3: kernel = k_gemm_tc<EPI_FUSED_ALLREDUCE, true>; smem = Cfg<EPI_FUSED_ALLREDUCE, true>::SMEM_BYTES;
            threads = Cfg<EPI_FUSED_ALLREDUCE, true>::THREADS; break;
    case 5: kernel = k_gemm_tc<EPI_ADD, false>; smem = Cfg<EPI_ADD, false>::SMEM_BYTES;
            threads = Cfg<EPI_ADD, false>::THREADS; break;
    default: kernel = k_gemm_tc<EPI_ADD, true>; smem = Cfg<EPI_ADD, true>::SMEM_BYTES;
             threads = Cfg<EPI_ADD, true>::THREADS; break;
  }
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !smem_configured[variant][dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    smem_configured[variant][dev].store(true, std::memory_order_release);
  }
  // A-views are used with the A box and B-views with the B box; a view used
  // on both sides gets two maps.
  std::unique_ptr<TcPrepared> prep(new TcPrepared);
  prep->kernel = kernel;
  prep->smem = smem;
  prep->threads = threads;
  cudaError_t status = cudaSuccess;
  size_t j = 0;
  const int fmt = plan.in_dtype == COCO_BF16 ? 1 : 0;
  // instruction descriptor: f32 accumulator, A and B of the input type, A K-major, B N-major,
  // N = 256, M = 128 per CTA (256 for the pair MMA)
  const uint32_t mma_m = two_sm && !bs ? 2 * BM : BM;
  const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (0u << 15) | (1u << 16) |
                         (static_cast<uint32_t>(BN >> 3) << 17) | ((mma_m >> 4) << 24);
  while (j < plan.jobs.size() && status == cudaSuccess) {
    std::unique_ptr<TcParams> Pown(new TcParams);
    TcParams* P = Pown.get();
    memset(P, 0, sizeof(TcParams));
    std::vector<int> amap(plan.views.size(), -1), bmap(plan.views.size(), -1);
    std::vector<std::pair<int, int>> orange;  // (first output, count) ranges already in this launch
    std::vector<int> obase;
    int nmaps = 0, nsegs = 0, nouts = 0, njobs = 0, tiles = 0;
    while (j < plan.jobs.size() && njobs < MAX_JOBS) {
      const Job& J = plan.jobs[j];
      // resources this job needs beyond what the launch already has
      int need_maps = 0;
      for (int k = 0; k < J.nseg; ++k) {
        const Seg& S = plan.segs[J.seg0 + k];
        need_maps += amap[S.a] < 0;
        need_maps += bmap[S.b] < 0;
      }
      int found = -1;
      for (size_t q = 0; q < orange.size(); ++q)
        if (orange[q].first == J.out && orange[q].second == J.nout) found = obase[q];
      const int need_out = (found < 0 ? J.nout : 0) + ((far || add) && J.res ? 1 : 0);
      if (nmaps + need_maps > MAX_MAPS || nsegs + J.nseg > MAX_SEGS || nouts + need_out > MAX_OUTS) break;
      Job nj = J;
      nj.seg0 = static_cast<int16_t>(nsegs);
      for (int k = 0; k < J.nseg; ++k) {
        Seg S = plan.segs[J.seg0 + k];
        if (amap[S.a] < 0) {
          if (!encode_view(&P->maps[nmaps], plan.views[S.a], plan.in_dtype, true)) { status = cudaErrorInvalidValue; break; }
          amap[S.a] = nmaps++;
        }
        if (bmap[S.b] < 0) {
          if (!encode_view(&P->maps[nmaps], plan.views[S.b], plan.in_dtype, false)) { status = cudaErrorInvalidValue; break; }
          bmap[S.b] = nmaps++;
        }
        S.a = static_cast<int16_t>(amap[S.a]);
        S.b = static_cast<int16_t>(bmap[S.b]);
        P->segs[nsegs++] = S;
      }
      if (status != cudaSuccess) break;
      if (found < 0) {  // the job's replicas get consecutive output slots
        found = nouts;
        for (int o = 0; o < J.nout && status == cudaSuccess; ++o) {
          P->outs[nouts] = plan.outs[J.out + o];
          if (!encode_out(&P->omaps[nouts], plan.outs[J.out + o], plan.out_dtype)) status = cudaErrorInvalidValue;
          ++nouts;
        }
        if (status != cudaSuccess) break;
        orange.emplace_back(J.out, J.nout);
        obase.push_back(found);
      }
      nj.out = found;
      nj.res_map = -1;
      if ((far || add) && J.res) {  // the residual / addend has the output's shape: a map like the outputs'
        OutView rv = plan.outs[J.out];
        rv.ptr = const_cast<void*>(J.res);
        if (!encode_out(&P->omaps[nouts], rv, plan.out_dtype)) { status = cudaErrorInvalidValue; break; }
        nj.res_map = static_cast<int16_t>(nouts++);
      }
      nj.kblocks = 0;
      for (int k = 0; k < J.nseg; ++k) nj.kblocks += (plan.segs[J.seg0 + k].klen + BK - 1) / BK;
      if (nj.kblocks <= 0) { status = cudaErrorInvalidValue; break; }  // an empty contraction is zero-filled, not run
      P->jobs[njobs] = nj;
      P->unit_start[njobs] = tiles;
      if (bs)  // units of up to BS_MTILES m-tiles sharing one B tile
        tiles += J.nb * ((J.m + BS_MTILES * BM - 1) / (BS_MTILES * BM)) * ((J.n + BN - 1) / BN);
      else  // units of two vertically adjacent tiles, one per CTA of the pair
        tiles += J.nb * ((J.m + 2 * BM - 1) / (2 * BM)) * ((J.n + BN - 1) / BN);
      ++njobs;
      ++j;
    }
    if (status != cudaSuccess) break;
    if (njobs == 0) { status = cudaErrorInvalidValue; break; }  // a single job exceeds the limits
    P->unit_start[njobs] = tiles;
    P->njobs = njobs;
    {
      // Long k-loops (64 or more k-blocks) whose largest whole B operand fits in half of L2 walk
      // each job one pair of m-tiles at a time across all its n-tiles: B stays in L2 while A
      // streams past once, which cut DRAM reads and, under the power cap, bought clock (case 1:
      // 1% faster sustained). Otherwise groups of GROUP_M m-tiles share both operands' slices
      // within a wave (1% faster on the K = 512 MatMul).
      int64_t bmax = 0;
      int kbmin = 1 << 30;
      for (int q = 0; q < njobs; ++q) {
        int64_t b = 0;
        for (int k = 0; k < P->jobs[q].nseg; ++k)
          b += static_cast<int64_t>(P->segs[P->jobs[q].seg0 + k].klen) * P->jobs[q].n * 2;
        bmax = b > bmax ? b : bmax;
        kbmin = P->jobs[q].kblocks < kbmin ? P->jobs[q].kblocks : kbmin;
      }
      P->group_pairs = (bmax <= (int64_t(64) << 20) && kbmin >= 64) ? 1 : GROUP_M / 2;
      // the grouped raster on long k-loops re-reads operands from DRAM when the pairs of a wave drift
      // apart; the pair-MMA launch then keeps its producers in step (a cooperative launch)
      P->wave_sync = (two_sm && !bs && P->group_pairs != 1 && kbmin >= 64) ? 1 : 0;
    }
    P->total_units = tiles;
    P->idesc = idesc;
    P->out_dtype = plan.out_dtype;
    P->err = nullptr;  // set per launch
    P->bias = plan.far.bias;
    P->seed = plan.far.seed;
    P->keep_threshold = plan.far.keep_threshold;
    P->scale = plan.far.scale;
    P->dropout = plan.far.dropout ? 1 : 0;
    const int pairs = sm_count() / 2;  // persistent: one CTA pair per two SMs (B-stationary: one CTA per SM)
    prep->grids.push_back(bs ? (tiles < sm_count() ? tiles : sm_count()) : 2 * (tiles < pairs ? tiles : pairs));
    prep->params.push_back(std::move(Pown));
  }
  if (status != cudaSuccess) return status;
  *out = prep.release();
  return cudaSuccess;
}

cudaError_t tc_launch(TcPrepared* prep, cudaStream_t s, unsigned int* err_word) {
  cudaError_t status = cudaSuccess;
  for (size_t i = 0; i < prep->params.size() && status == cudaSuccess; ++i) {
    TcParams* P = prep->params[i].get();
    const int grid = prep->grids[i];
    P->err = err_word;
    const int32_t want_sync = P->wave_sync;
    bool launched = false;
    if (want_sync) {
      void* base = nullptr;
      if (cudaGetSymbolAddress(&base, g_wave_counters) == cudaSuccess) {
        P->wave_counter = static_cast<unsigned int*>(base) + (g_wave_slot.fetch_add(1) % kWaveSlots);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(prep->threads);
        cfg.dynamicSmemBytes = prep->smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: they wait on each other
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaMemsetAsync(P->wave_counter, 0, sizeof(unsigned int), s) == cudaSuccess &&
            cudaLaunchKernelEx(&cfg, prep->kernel, *P) == cudaSuccess)
          launched = true;
      }
      (void)cudaGetLastError();  // a refused cooperative launch falls back to the plain one below
    }
    if (!launched) {
      P->wave_sync = 0;  // the block is copied at launch: the prepared request is restored below
      prep->kernel<<<grid, prep->threads, prep->smem, s>>>(*P);
      P->wave_sync = want_sync;
    }
    count_launch();
    status = cudaGetLastError();
  }
  return status;
}

cudaError_t launch_gemm_tc(const GemmPlan& plan, cudaStream_t s, unsigned int* err_word) {
  TcPrepared* prep = nullptr;
  cudaError_t e = tc_prepare(plan, &prep);
  if (e != cudaSuccess) return e;
  e = tc_launch(prep, s, err_word);
  tc_free(prep);
  return e;
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t s, unsigned int* err_word) {
  k_wait_selftest<<<1, 64, 0, s>>>(err_word, timeout_ns);
  count_launch();
  return cudaGetLastError();
}

}  // namespace coco
