// coco_allreduce_rs_ag_noalloc: AllReduce split into ReduceScatter + AllGather
// for callers that cannot allocate device memory, with the sliced
// intermediate kept in a fixed array that is part of the library image.
//
// Who needs it: code that must not call cudaMalloc (or any allocator) once it
// is running -- for example a latency-critical loop where an allocation could
// stall or fail in the middle of a step, or a plug-in embedded in a host
// application that owns all device memory and gives the plug-in no allocator.
// Such a caller passes only the inputs and outputs; the scratch lives in
// `g_rs_ag_scratch` below.
//
// Costs and limits, stated for users:
//   * every GPU that loads libcoco.so holds kNoAllocScratchBytes (16 MiB) of
//     device memory for this array until the process exits;
//   * one call needs ngroups * numel * element size bytes of it (the N slices
//     of every group); larger requests return COCO_ERR_UNSUPPORTED and
//     launch nothing;
//   * every call shares the one array, so calls whose kernels can overlap on
//     the GPU (different streams without ordering between them, or several
//     host threads) race on it; calls ordered on one stream are safe;
//   * the array keeps whatever the last call left in it; nothing has to start
//     at zero because the ReduceScatter writes every scratch element before
//     the AllGather reads it.
//
// Set-up: the first call on each device (with that device current) resolves
// the device address of the array with cudaGetSymbolAddress and caches it,
// together with the identity of the CUDA context it belongs to; later calls in
// the same context reuse the address. A new context on the device (after
// cudaDeviceReset, for example) gets the array at a new address, so a call that
// finds a different context resolves it again. Make the first call on a device
// (and the first after a reset) before any stream capture: a call that needs
// the set-up while its stream is being captured returns COCO_ERR_UNSUPPORTED
// and launches nothing.

#include <cuda.h>

#include <mutex>

#include "coco.h"
#include "internal.h"

#define COCO_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr size_t kSliceAlign = 256;

// In host code this name is only a stand-in for the device symbol; its device
// address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_rs_ag_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchSlot {
  unsigned long long ctx_id;  // the context the address belongs to (0: none cached)
  void* addr;
};
ScratchSlot g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (driver entry points
// looked up once through the runtime), or 0 when there is none or the driver
// cannot tell.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

enum SetupResult { kSetupOk, kSetupUnderCapture, kSetupCudaError };

// Device address of the scratch array in the current context of the current
// device, resolved once per context. The resolution is refused while
// `stream` is being captured.
SetupResult scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kSetupCudaError;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const unsigned long long ctx = current_context_id();
  if (g_scratch[dev].addr && ctx != 0 && g_scratch[dev].ctx_id == ctx) {
    *out = g_scratch[dev].addr;
    return kSetupOk;
  }
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capturing) != cudaSuccess) {
    (void)cudaGetLastError();
    return kSetupCudaError;
  }
  if (capturing != cudaStreamCaptureStatusNone) return kSetupUnderCapture;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_rs_ag_scratch) != cudaSuccess || !p) {
    (void)cudaGetLastError();
    return kSetupCudaError;
  }
  // the context exists now (the lookup initialises it); an unknown id caches nothing
  g_scratch[dev].ctx_id = current_context_id();
  g_scratch[dev].addr = g_scratch[dev].ctx_id ? p : nullptr;
  *out = p;
  return kSetupOk;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// The extent rule of the library's other entry points: every dimension and
// the per-rank element count at most 2^40, checked before any product can
// overflow.
constexpr int64_t kMaxElems = int64_t(1) << 40;

}  // namespace

COCO_EXPORT coco_status coco_allreduce_rs_ag_noalloc(const coco_tensor* in, const coco_tensor* out, void* stream) {
  // Structural checks first, so malformed requests fail before any CUDA call.
  if (!in || !out) return COCO_ERR_NULL;
  if (in->dtype < COCO_F32 || in->dtype > COCO_BF16 || out->dtype != in->dtype) return COCO_ERR_DTYPE;
  if (in->layout != COCO_LOCAL || out->layout != COCO_REPLICATED) return COCO_ERR_LAYOUT;
  if (in->ndim < 1 || in->ndim > COCO_MAX_DIMS || out->ndim != in->ndim) return COCO_ERR_SHAPE;
  if (in->nranks < 1 || in->ngroups < 1 || static_cast<int64_t>(in->nranks) * in->ngroups > COCO_MAX_PTRS)
    return COCO_ERR_SHAPE;
  if (out->nranks != in->nranks || out->ngroups != in->ngroups) return COCO_ERR_SHAPE;
  int64_t numel = 1;
  for (int d = 0; d < in->ndim; ++d) {
    if (in->shape[d] < 0 || in->shape[d] > kMaxElems || in->shape[d] != out->shape[d]) return COCO_ERR_SHAPE;
    if (in->shape[d] != 0 && numel > kMaxElems / in->shape[d]) return COCO_ERR_SHAPE;
    numel *= in->shape[d];
  }
  if (in->shape[0] % in->nranks) return COCO_ERR_SHAPE;  // the scratch splits dimension 0
  if (numel == 0) return COCO_OK;
  const size_t esize = static_cast<size_t>(coco::dtype_size(in->dtype));
  const size_t slice_bytes = round_up(static_cast<size_t>(numel / in->nranks) * esize, kSliceAlign);
  const size_t need = slice_bytes * static_cast<size_t>(in->nranks) * static_cast<size_t>(in->ngroups);
  if (need > kNoAllocScratchBytes) return COCO_ERR_UNSUPPORTED;

  void* base = nullptr;
  switch (scratch_address(static_cast<cudaStream_t>(stream), &base)) {
    case kSetupOk: break;
    case kSetupUnderCapture: return COCO_ERR_UNSUPPORTED;
    default: return COCO_ERR_CUDA;
  }

  // The scratch as a caller would have passed it: SLICED on dimension 0, one
  // 256-byte-aligned slice per (group, rank).
  coco_tensor scratch = *in;
  scratch.layout = COCO_SLICED;
  scratch.slice_dim = 0;
  for (int i = 0; i < in->nranks * in->ngroups; ++i)
    scratch.ptr[i] = static_cast<unsigned char*>(base) + static_cast<size_t>(i) * slice_bytes;
  for (int i = in->nranks * in->ngroups; i < COCO_MAX_PTRS; ++i) scratch.ptr[i] = nullptr;
  return coco_allreduce_rs_ag(in, &scratch, out, stream);
}
