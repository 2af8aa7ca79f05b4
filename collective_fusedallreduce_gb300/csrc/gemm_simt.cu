// fp32 GEMM on the FMA units, driven by the same job / K-segment plan as the
// tensor-core kernel. It serves fp32 operands, where the 1e-5 relative
// tolerance rules out tf32 tensor-core arithmetic.
//
// [Decomp] "Overlap Communication with Dependent Computation via
// Decomposition in Large Deep Learning Models", §5.1: the K-segments of a job
// are visited in the ring order the planner wrote them, so the fp32
// accumulation follows the order in which the looped collective adds partial
// results.
//
// Tile 64 x 64 x 16, 256 threads, 4 x 4 outputs per thread, operands staged in
// shared memory with bounds checks on every element (any shape, any offset).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace coco {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;
constexpr int MAX_VIEWS = 128, MAX_JOBS = 128, MAX_SEGS = 256, MAX_OUTS = 64;

struct SimtParams {
  View views[MAX_VIEWS];
  Job jobs[MAX_JOBS];
  Seg segs[MAX_SEGS];
  OutView outs[MAX_OUTS];
  int32_t tile_start[MAX_JOBS + 1];
  int32_t njobs, total_tiles, out_dtype;
  int32_t accumulate;  // EPI_ADD: out (fp32) += the product
};
static_assert(sizeof(SimtParams) <= 32000, "kernel parameter block too large");

__device__ __forceinline__ float load_f32(const View& v, int64_t b, int64_t r, int64_t c) {
  if (b < 0 || b >= v.nb || r < 0 || r >= v.rows || c < 0 || c >= v.cols) return 0.0f;
  return static_cast<const float*>(v.ptr)[b * v.bstride + r * v.ld + c];
}

__global__ void __launch_bounds__(256) k_gemm_simt(const __grid_constant__ SimtParams P) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int t = blockIdx.x; t < P.total_tiles; t += gridDim.x) {
    int j = 0;
    while (j + 1 < P.njobs && P.tile_start[j + 1] <= t) ++j;
    const Job& J = P.jobs[j];
    const int mtiles = (J.m + TM - 1) / TM, ntiles = (J.n + TN - 1) / TN;
    const int local = t - P.tile_start[j];
    const int bb = local / (mtiles * ntiles);
    const int rem = local - bb * mtiles * ntiles;
    const int mt = rem / ntiles, nt = rem % ntiles;
    float acc[4][4] = {};
    for (int si = 0; si < J.nseg; ++si) {
      const Seg& S = P.segs[J.seg0 + si];
      const View& A = P.views[S.a];
      const View& B = P.views[S.b];
      for (int k0 = 0; k0 < S.klen; k0 += TK) {
        for (int i = threadIdx.x; i < TM * TK; i += 256) {
          const int kk = i % TK, mm = i / TK;
          const int k = k0 + kk;
          As[kk][mm] = k < S.klen ? load_f32(A, S.a_b0 + bb, S.a_r0 + mt * TM + mm, S.a_k0 + k) : 0.0f;
        }
        for (int i = threadIdx.x; i < TN * TK; i += 256) {
          const int nn = i % TN, kk = i / TN;
          const int k = k0 + kk;
          Bs[kk][nn] = k < S.klen ? load_f32(B, S.b_b0 + bb, S.b_k0 + k, S.b_c0 + nt * TN + nn) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
          float a[4], b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
          for (int i = 0; i < 4; ++i) b[i] = Bs[kk][tx * 4 + i];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(a[i], b[q], acc[i][q]);
        }
        __syncthreads();
      }
    }
    const OutView& O = P.outs[J.out];
    for (int i = 0; i < 4; ++i) {
      const int row = mt * TM + ty * 4 + i;
      if (row >= J.m) continue;
      for (int q = 0; q < 4; ++q) {
        const int col = nt * TN + tx * 4 + q;
        if (col >= J.n) continue;
        const int64_t off = static_cast<int64_t>(J.o_b0 + bb) * O.bstride + static_cast<int64_t>(J.o_r0 + row) * O.ld +
                            (J.o_c0 + col);
        if (P.out_dtype == COCO_F32) {
          float* o = static_cast<float*>(O.ptr) + off;
          *o = P.accumulate ? *o + acc[i][q] : acc[i][q];
        }
        else if (P.out_dtype == COCO_F16) static_cast<__half*>(O.ptr)[off] = __float2half_rn(acc[i][q]);
        else static_cast<__nv_bfloat16*>(O.ptr)[off] = __float2bfloat16_rn(acc[i][q]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmPlan& plan, cudaStream_t s) {
  SimtParams* P = new SimtParams;
  cudaError_t status = cudaSuccess;
  size_t j = 0;
  while (j < plan.jobs.size() && status == cudaSuccess) {
    memset(P, 0, sizeof(SimtParams));
    std::vector<int> vmap(plan.views.size(), -1), omap(plan.outs.size(), -1);
    int nviews = 0, nsegs = 0, nouts = 0, njobs = 0, tiles = 0;
    while (j < plan.jobs.size() && njobs < MAX_JOBS) {
      const Job& J = plan.jobs[j];
      int need = 0;
      for (int k = 0; k < J.nseg; ++k) {
        const Seg& S = plan.segs[J.seg0 + k];
        need += vmap[S.a] < 0;
        need += (vmap[S.b] < 0 && S.b != S.a);
      }
      const int need_out = omap[J.out] < 0;
      if (nviews + need > MAX_VIEWS || nsegs + J.nseg > MAX_SEGS || nouts + need_out > MAX_OUTS) break;
      Job nj = J;
      nj.seg0 = static_cast<int16_t>(nsegs);
      for (int k = 0; k < J.nseg; ++k) {
        Seg S = plan.segs[J.seg0 + k];
        if (vmap[S.a] < 0) { P->views[nviews] = plan.views[S.a]; vmap[S.a] = nviews++; }
        if (vmap[S.b] < 0) { P->views[nviews] = plan.views[S.b]; vmap[S.b] = nviews++; }
        S.a = static_cast<int16_t>(vmap[S.a]);
        S.b = static_cast<int16_t>(vmap[S.b]);
        P->segs[nsegs++] = S;
      }
      if (omap[J.out] < 0) { P->outs[nouts] = plan.outs[J.out]; omap[J.out] = nouts++; }
      nj.out = omap[J.out];
      P->jobs[njobs] = nj;
      P->tile_start[njobs] = tiles;
      tiles += J.nb * ((J.m + TM - 1) / TM) * ((J.n + TN - 1) / TN);
      ++njobs;
      ++j;
    }
    if (njobs == 0) { status = cudaErrorInvalidValue; break; }
    P->tile_start[njobs] = tiles;
    P->njobs = njobs;
    P->total_tiles = tiles;
    P->out_dtype = plan.out_dtype;
    P->accumulate = plan.mode == EPI_ADD ? 1 : 0;
    const int cap = sm_count() * 4;
    k_gemm_simt<<<tiles < cap ? tiles : cap, 256, 0, s>>>(*P);
    count_launch();
    status = cudaGetLastError();
  }
  delete P;
  return status;
}

}  // namespace coco
