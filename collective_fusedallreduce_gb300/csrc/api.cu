// C-ABI of libcoco: argument validation, shard-schedule planning and
// dispatch to the kernels. Every entry point validates everything on the host
// before its first CUDA call.
//
// Layout semantics: [CoCoNet] "Breaking the Computation and Communication
// Abstraction Barrier in Distributed Machine Learning Workloads" (sliced /
// replicated / local tensors and the layout rules of its Fig. 3 program).
// Looped schedules: [Decomp] "Overlap Communication with Dependent
// Computation via Decomposition in Large Deep Learning Models", §5.1.

#include <atomic>
#include <algorithm>
#include <list>
#include <memory>
#include <mutex>
#include <set>
#include <cmath>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "coco.h"
#include "internal.h"

#define COCO_EXPORT extern "C" __attribute__((visibility("default")))

using namespace coco;

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};

coco_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return COCO_OK;
  g_last_cuda_error = static_cast<int>(e);
  return COCO_ERR_CUDA;
}

// ------------------------------------------------------------ validation

struct TInfo {
  int dtype = 0, layout = 0, ndim = 0, slice_dim = -1, nranks = 0, ngroups = 0;
  int64_t shape[COCO_MAX_DIMS] = {0, 0, 0};  // as given
  int64_t local[COCO_MAX_DIMS] = {0, 0, 0};  // per-rank
  int64_t numel = 0;                         // per rank
  int64_t bytes = 0;                         // per rank
  const coco_tensor* t = nullptr;
  void* ptr(int g, int r) const { return t->ptr[g * nranks + r]; }
};

coco_status check_tensor(const coco_tensor* t, TInfo* o) {
  if (!t) return COCO_ERR_NULL;
  if (t->dtype < COCO_F32 || t->dtype > COCO_BF16) return COCO_ERR_DTYPE;
  if (t->layout < COCO_LOCAL || t->layout > COCO_REPLICATED) return COCO_ERR_LAYOUT;
  if (t->ndim < 1 || t->ndim > COCO_MAX_DIMS) return COCO_ERR_SHAPE;
  if (t->nranks < 1 || t->ngroups < 1 || static_cast<int64_t>(t->nranks) * t->ngroups > COCO_MAX_PTRS)
    return COCO_ERR_SHAPE;
  o->t = t;
  o->dtype = t->dtype;
  o->layout = t->layout;
  o->ndim = t->ndim;
  o->nranks = t->nranks;
  o->ngroups = t->ngroups;
  o->numel = 1;
  for (int d = 0; d < t->ndim; ++d) {
    if (t->shape[d] < 0 || t->shape[d] > (int64_t(1) << 40)) return COCO_ERR_SHAPE;
    o->shape[d] = o->local[d] = t->shape[d];
  }
  if (t->layout == COCO_SLICED) {
    if (t->slice_dim < 0 || t->slice_dim >= t->ndim) return COCO_ERR_SHAPE;
    if (t->shape[t->slice_dim] % t->nranks) return COCO_ERR_SHAPE;  // "equally distributed"
    o->slice_dim = t->slice_dim;
    o->local[t->slice_dim] /= t->nranks;
  }
  // at most 2^40 elements per rank (far beyond any device's memory), so no size below overflows
  for (int d = 0; d < t->ndim; ++d) {
    if (o->local[d] != 0 && o->numel > (int64_t(1) << 40) / o->local[d]) return COCO_ERR_SHAPE;
    o->numel *= o->local[d];
  }
  o->bytes = o->numel * dtype_size(t->dtype);
  if (o->numel == 0) return COCO_OK;
  for (int i = 0; i < t->nranks * t->ngroups; ++i) {
    if (!t->ptr[i]) return COCO_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(t->ptr[i]) & 15) return COCO_ERR_ALIGN;
  }
  if (o->local[t->ndim - 1] % 8) return COCO_ERR_ALIGN;
  return COCO_OK;
}

bool same_ranks(const TInfo& a, const TInfo& b) { return a.nranks == b.nranks && a.ngroups == b.ngroups; }

bool same_local_shape(const TInfo& a, const TInfo& b) {
  if (a.ndim != b.ndim) return false;
  for (int d = 0; d < a.ndim; ++d)
    if (a.local[d] != b.local[d]) return false;
  return true;
}

struct Range {
  uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range range_of(const void* p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + static_cast<uintptr_t>(bytes)};
}

// Outputs must not partially overlap each other or any input. `exact_ok`:
// an output may coincide exactly with an input (element-wise kernels read
// every input element before writing the outputs at the same index).
coco_status check_alias(const std::vector<Range>& outs, const std::vector<Range>& ins, bool exact_ok) {
  for (size_t i = 0; i < outs.size(); ++i) {
    for (size_t j = i + 1; j < outs.size(); ++j) {
      if (outs[i].lo == outs[j].lo && outs[i].hi == outs[j].hi) continue;  // the same buffer: written once
      if (overlap(outs[i], outs[j])) return COCO_ERR_ALIAS;
    }
    for (const Range& r : ins) {
      if (!overlap(outs[i], r)) continue;
      if (exact_ok && outs[i].lo == r.lo && outs[i].hi == r.hi) continue;
      return COCO_ERR_ALIAS;
    }
  }
  return COCO_OK;
}

// Distinct output pointers of every group, compacted into tables.out.
void fill_outputs(const TInfo& out, ReduceTables* t) {
  for (int g = 0; g < out.ngroups; ++g) {
    int n = 0;
    for (int r = 0; r < out.nranks; ++r) {
      void* p = out.ptr(g, r);
      bool seen = false;
      for (int q = 0; q < n; ++q) seen |= (t->out[g * out.nranks + q] == p);
      if (!seen) t->out[g * out.nranks + n++] = p;
    }
    t->nout[g] = n;
  }
}

void tensor_ranges(const TInfo& a, std::vector<Range>* v, bool first_only = false) {
  if (a.bytes == 0) return;
  for (int g = 0; g < a.ngroups; ++g)
    for (int r = 0; r < (first_only ? 1 : a.nranks); ++r) v->push_back(range_of(a.ptr(g, r), a.bytes));
}

// ---------------------------------------------------------- einsum specs

struct Spec {
  bool batched = false;
  // label positions: lhs [b] m k, rhs [b] k n, out [b] m n
};

bool parse_spec(const char* spec, Spec* s) {
  if (!spec) return false;
  std::string x;
  for (const char* p = spec; *p; ++p)
    if (*p != ' ') x.push_back(*p);
  if (x == "mk,kn->mn") { s->batched = false; return true; }
  if (x == "bmk,bkn->bmn") { s->batched = true; return true; }
  return false;
}

// Label of dimension d of an operand: 'b', 'm', 'k' (lhs) / 'b', 'k', 'n' (rhs).
char label(const Spec& s, bool is_lhs, int d) {
  const char* l = s.batched ? (is_lhs ? "bmk" : "bkn") : (is_lhs ? "mk" : "kn");
  return l[d];
}

struct Dims3 {
  int64_t b, r, c;  // batch, rows, cols of a per-rank operand
};
Dims3 dims_of(const Spec& s, const int64_t* ext) {
  return s.batched ? Dims3{ext[0], ext[1], ext[2]} : Dims3{1, ext[0], ext[1]};
}

bool fits_i32(int64_t v) { return v >= 0 && v < (int64_t(1) << 31); }

View make_view(const void* p, Dims3 d) {
  View v;
  v.ptr = p;
  v.nb = static_cast<int32_t>(d.b);
  v.rows = static_cast<int32_t>(d.r);
  v.cols = static_cast<int32_t>(d.c);
  v.ld = d.c;
  v.bstride = d.r * d.c;
  return v;
}

OutView make_out(void* p, Dims3 d) {
  OutView o;
  o.ptr = p;
  o.ld = d.c;
  o.bstride = d.r * d.c;
  o.nb = static_cast<int32_t>(d.b);
  o.rows = static_cast<int32_t>(d.r);
  o.cols = static_cast<int32_t>(d.c);
  return o;
}

int add_view(GemmPlan* P, const View& v) {
  for (size_t i = 0; i < P->views.size(); ++i) {
    const View& w = P->views[i];
    if (w.ptr == v.ptr && w.nb == v.nb && w.rows == v.rows && w.cols == v.cols && w.ld == v.ld &&
        w.bstride == v.bstride)
      return static_cast<int>(i);
  }
  P->views.push_back(v);
  return static_cast<int>(P->views.size() - 1);
}

int add_out(GemmPlan* P, const OutView& o) {
  for (size_t i = 0; i < P->outs.size(); ++i)
    if (P->outs[i].ptr == o.ptr) return static_cast<int>(i);
  P->outs.push_back(o);
  return static_cast<int>(P->outs.size() - 1);
}

Seg make_seg(int a, int b, int64_t klen) {
  Seg s;
  std::memset(&s, 0, sizeof(s));
  s.a = static_cast<int16_t>(a);
  s.b = static_cast<int16_t>(b);
  s.klen = static_cast<int32_t>(klen);
  return s;
}

Job make_job(int out, Dims3 ext) {
  Job j;
  std::memset(&j, 0, sizeof(j));
  j.out = out;
  j.nout = 1;
  j.nb = static_cast<int32_t>(ext.b);
  j.m = static_cast<int32_t>(ext.r);
  j.n = static_cast<int32_t>(ext.c);
  return j;
}

// Zero-fills every output of a plan whose contraction length is 0.
coco_status zero_outputs(const TInfo& out, cudaStream_t s) {
  for (int g = 0; g < out.ngroups; ++g)
    for (int r = 0; r < out.nranks; ++r) {
      cudaError_t e = cudaMemsetAsync(out.ptr(g, r), 0, out.bytes, s);
      if (e != cudaSuccess) return cuda_status(e);
    }
  return COCO_OK;
}

// Host-side TMA rules for the tensor-core path: 16-byte aligned view bases
// and x coordinates (elements x 2 bytes a multiple of 16), 16-byte strides.
bool tma_ok(const GemmPlan& P) {
  for (const View& v : P.views) {
    if (reinterpret_cast<uintptr_t>(v.ptr) & 15) return false;
    if ((v.ld * 2) % 16 || (v.bstride * 2) % 16) return false;
  }
  for (const Seg& s : P.segs)
    if (s.a_k0 % 8 || s.b_c0 % 8) return false;
  for (const Job& j : P.jobs)
    if (j.o_c0 % 8) return false;
  return true;
}

coco_status run_plan(const GemmPlan& P, cudaStream_t s) {
  if (P.jobs.empty()) return COCO_OK;
  if (P.in_dtype == COCO_F32) return cuda_status(launch_gemm_simt(P, s));
  if (!tma_ok(P)) return COCO_ERR_ALIGN;
  unsigned int* err = gemm_error_word();
  if (!err) return cuda_status(cudaErrorSymbolNotFound);
  cudaError_t e = launch_gemm_tc(P, s, err);
  if (e == cudaErrorNotSupported) return COCO_ERR_UNSUPPORTED;
  return cuda_status(e);
}

// ------------------------------------------------------------ plan cache
//
// A call's plan (validated, with its tensor maps encoded) depends only on its
// arguments: the entry point, the spec and schedule, the fields of every
// coco_tensor argument that are in use (dtype, layout, shape, slice dim, rank
// and group counts, pointers), the fused epilogue's scalars and the current
// device. The cache keys each plan on exactly those, so a call that repeats
// them (a training loop calling the same shapes every step) skips
// validation, planning and tensor-map encoding. Only calls that passed
// validation are entered, and the device is read (a CUDA call) only for
// arguments that match an entry or have just passed validation, so invalid
// arguments are still refused before any CUDA call. The stream is not part
// of a plan. Least recently used entries beyond kPlanCacheSize are dropped.
constexpr size_t kPlanCacheSize = 64;

struct PlanKey {
  std::vector<uint64_t> w;
  bool ok = true;  // false: the arguments cannot be keyed (left to validation)
  explicit PlanKey(uint64_t entry) {
    w.reserve(256);
    w.push_back(entry);
  }
  void add(uint64_t v) { w.push_back(v); }
  void f32(float v) {
    uint32_t b;
    std::memcpy(&b, &v, 4);
    w.push_back(b);
  }
  void str(const char* s) {
    if (!s) { ok = false; return; }
    uint64_t word = 0;
    int i = 0;
    for (; s[i] && i < 64; ++i) {
      word = (word << 8) | static_cast<uint8_t>(s[i]);
      if ((i & 7) == 7) { w.push_back(word); word = 0; }
    }
    if (s[i]) { ok = false; return; }  // longer than any spec the library takes
    w.push_back(word);
    w.push_back(static_cast<uint64_t>(i));
  }
  void tensor(const coco_tensor* t) {
    if (!t) { w.push_back(~0ull); return; }
    if (t->ndim < 1 || t->ndim > COCO_MAX_DIMS || t->nranks < 1 || t->ngroups < 1 ||
        static_cast<int64_t>(t->nranks) * t->ngroups > COCO_MAX_PTRS) {
      ok = false;
      return;
    }
    w.push_back((static_cast<uint64_t>(static_cast<uint32_t>(t->dtype)) << 32) | static_cast<uint32_t>(t->layout));
    w.push_back((static_cast<uint64_t>(static_cast<uint32_t>(t->ndim)) << 32) | static_cast<uint32_t>(t->slice_dim));
    w.push_back((static_cast<uint64_t>(static_cast<uint32_t>(t->nranks)) << 32) | static_cast<uint32_t>(t->ngroups));
    for (int d = 0; d < t->ndim; ++d) w.push_back(static_cast<uint64_t>(t->shape[d]));
    for (int i = 0; i < t->nranks * t->ngroups; ++i) w.push_back(reinterpret_cast<uintptr_t>(t->ptr[i]));
  }
};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return dev;
}

struct PlanEntry {
  std::vector<uint64_t> key;
  int device = -1;
  GemmPlan plan;
  bool tma_ok = false;
  std::mutex m;  // launches of one entry set the per-launch fields of its parameter blocks
  TcPrepared* tc = nullptr;
  ~PlanEntry() {
    if (tc) tc_free(tc);
  }
};

class PlanCache {
 public:
  std::shared_ptr<PlanEntry> find(const std::vector<uint64_t>& key) {
    std::lock_guard<std::mutex> g(m_);
    int dev = -2;  // read once, and only when the arguments match an entry
    for (auto it = lru_.begin(); it != lru_.end(); ++it)
      if ((*it)->key == key && (*it)->device == (dev == -2 ? (dev = current_device()) : dev)) {
        if (it != lru_.begin()) lru_.splice(lru_.begin(), lru_, it);
        hits_.fetch_add(1, std::memory_order_relaxed);
        return lru_.front();
      }
    misses_.fetch_add(1, std::memory_order_relaxed);
    return nullptr;
  }
  std::shared_ptr<PlanEntry> insert(std::vector<uint64_t> key, GemmPlan&& plan, bool tma) {
    auto e = std::make_shared<PlanEntry>();
    e->key = std::move(key);
    e->device = current_device();
    e->plan = std::move(plan);
    e->tma_ok = tma;
    std::lock_guard<std::mutex> g(m_);
    lru_.push_front(e);
    while (lru_.size() > kPlanCacheSize) lru_.pop_back();  // in-use entries live on in their callers
    return e;
  }
  void clear() {
    std::lock_guard<std::mutex> g(m_);
    lru_.clear();
  }
  void stats(uint64_t* hits, uint64_t* misses, uint64_t* entries) {
    std::lock_guard<std::mutex> g(m_);
    if (hits) *hits = hits_.load();
    if (misses) *misses = misses_.load();
    if (entries) *entries = lru_.size();
  }

 private:
  std::mutex m_;
  std::list<std::shared_ptr<PlanEntry>> lru_;  // most recently used first
  std::atomic<uint64_t> hits_{0}, misses_{0};
};

PlanCache& plan_cache() {
  static PlanCache* c = new PlanCache;  // never destroyed: calls may come during process exit
  return *c;
}

// Runs a cached plan: the fp32 path launches from the plan; the tensor-core path encodes its maps
// once (the first run of the entry) and relaunches the prepared parameter blocks after that.
coco_status run_entry(PlanEntry& e, cudaStream_t s) {
  const GemmPlan& P = e.plan;
  if (P.jobs.empty()) return COCO_OK;
  if (P.in_dtype == COCO_F32) return cuda_status(launch_gemm_simt(P, s));
  if (!e.tma_ok) return COCO_ERR_ALIGN;
  unsigned int* err = gemm_error_word();
  if (!err) return cuda_status(cudaErrorSymbolNotFound);
  std::lock_guard<std::mutex> g(e.m);
  if (!e.tc) {
    cudaError_t x = tc_prepare(P, &e.tc);
    if (x == cudaErrorNotSupported) return COCO_ERR_UNSUPPORTED;
    if (x != cudaSuccess) return cuda_status(x);
  }
  return cuda_status(tc_launch(e.tc, s, err));
}

// Enters a validated plan under `key` (when the call could be keyed) and runs it.
coco_status run_keyed(GemmPlan&& P, const PlanKey& key, cudaStream_t s) {
  if (!key.ok) return run_plan(P, s);
  const bool tma = P.in_dtype == COCO_F32 || tma_ok(P);
  std::shared_ptr<PlanEntry> e = plan_cache().insert(key.w, std::move(P), tma);
  return run_entry(*e, s);
}

// Output pointers of a group that need computing: every rank for LOCAL, the
// first rank of each distinct pointer for REPLICATED.
std::vector<int> output_ranks(const TInfo& out, int g) {
  std::vector<int> ranks;
  for (int r = 0; r < out.nranks; ++r) {
    bool seen = false;
    if (out.layout == COCO_REPLICATED)
      for (int q : ranks) seen |= out.ptr(g, q) == out.ptr(g, r);
    if (!seen) ranks.push_back(r);
  }
  return ranks;
}

coco_status einsum_alias(const TInfo& lhs, const TInfo& rhs, const TInfo& out) {
  std::vector<Range> outs, ins;
  tensor_ranges(out, &outs);
  tensor_ranges(lhs, &ins);
  tensor_ranges(rhs, &ins);
  return check_alias(outs, ins, false);
}

}  // namespace

// ================================================================ entries

COCO_EXPORT const char* coco_status_string(coco_status s) {
  switch (s) {
    case COCO_OK: return "COCO_OK";
    case COCO_ERR_NULL: return "COCO_ERR_NULL: a required pointer is NULL";
    case COCO_ERR_SHAPE: return "COCO_ERR_SHAPE: shapes or rank counts disagree, or a slice is uneven";
    case COCO_ERR_DTYPE: return "COCO_ERR_DTYPE: unknown dtype or operand dtypes disagree";
    case COCO_ERR_LAYOUT: return "COCO_ERR_LAYOUT: an operand has a layout the operation does not take";
    case COCO_ERR_ALIGN: return "COCO_ERR_ALIGN: pointer not 16-byte aligned or inner dim not a multiple of 8";
    case COCO_ERR_ALIAS: return "COCO_ERR_ALIAS: an output overlaps an input or another output";
    case COCO_ERR_UNSUPPORTED: return "COCO_ERR_UNSUPPORTED: not implemented by this library";
    case COCO_ERR_CUDA: return "COCO_ERR_CUDA: a CUDA call or kernel launch failed";
    case COCO_ERR_TIMEOUT: return "COCO_ERR_TIMEOUT: a bounded device-side wait gave up";
    case COCO_ERR_VALUE: return "COCO_ERR_VALUE: a scalar argument is out of range";
  }
  return "unknown coco_status";
}

COCO_EXPORT int coco_version(void) { return 100; }

COCO_EXPORT int coco_last_cuda_error(void) { return g_last_cuda_error; }

COCO_EXPORT uint64_t coco_kernel_launches(void) { return g_launches.load(); }

void coco::count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static coco_status fused_allreduce_impl(const coco_tensor* partials, const void* bias,
                                        const coco_tensor* residual, float dropout_p, uint64_t seed,
                                        uint64_t index_base, const coco_tensor* out, void* stream) {
  TInfo in, o, res;
  coco_status st;
  if ((st = check_tensor(partials, &in)) != COCO_OK) return st;
  if ((st = check_tensor(out, &o)) != COCO_OK) return st;
  if (in.layout != COCO_LOCAL || o.layout != COCO_REPLICATED) return COCO_ERR_LAYOUT;
  if (in.dtype != o.dtype) return COCO_ERR_DTYPE;
  if (!same_ranks(in, o) || !same_local_shape(in, o)) return COCO_ERR_SHAPE;
  if (residual) {
    if ((st = check_tensor(residual, &res)) != COCO_OK) return st;
    if (res.layout != COCO_REPLICATED) return COCO_ERR_LAYOUT;
    if (res.dtype != in.dtype) return COCO_ERR_DTYPE;
    if (!same_ranks(in, res) || !same_local_shape(in, res)) return COCO_ERR_SHAPE;
  }
  if (!(dropout_p >= 0.0f && dropout_p <= 1.0f)) return COCO_ERR_VALUE;  // also rejects NaN
  const int64_t H = in.local[in.ndim - 1];
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 15)) return COCO_ERR_ALIGN;
  if (index_base % static_cast<uint64_t>(16 / dtype_size(in.dtype))) return COCO_ERR_ALIGN;
  if (in.numel == 0) return COCO_OK;

  std::vector<Range> outs, ins;
  tensor_ranges(o, &outs);
  tensor_ranges(in, &ins);
  if (residual) tensor_ranges(res, &ins, true);
  if ((st = check_alias(outs, ins, true)) != COCO_OK) return st;
  if (bias) {
    const Range b = range_of(bias, H * dtype_size(in.dtype));
    for (const Range& r : outs)
      if (overlap(r, b)) return COCO_ERR_ALIAS;
  }

  FarLaunch L;
  std::memset(&L, 0, sizeof(L));
  for (int i = 0; i < in.nranks * in.ngroups; ++i) L.t.in[i] = partials->ptr[i];
  fill_outputs(o, &L.t);
  for (int g = 0; g < in.ngroups; ++g) L.t.residual[g] = residual ? res.ptr(g, 0) : nullptr;
  L.dtype = in.dtype;
  L.nranks = in.nranks;
  L.ngroups = in.ngroups;
  L.numel = in.numel;
  L.bias = bias;
  L.bias_len = H;
  L.dropout = dropout_p > 0.0f;
  const double keep = 1.0 - static_cast<double>(dropout_p);
  L.keep_threshold = static_cast<uint32_t>(std::floor(keep * 16777216.0));
  L.scale = dropout_p < 1.0f ? static_cast<float>(1.0 / keep) : 0.0f;
  L.seed = seed;
  L.index_base = index_base;
  return cuda_status(launch_fused_allreduce(L, static_cast<cudaStream_t>(stream)));
}

COCO_EXPORT coco_status coco_fused_allreduce(const coco_tensor* partials, const void* bias,
                                             const coco_tensor* residual, float dropout_p, uint64_t seed,
                                             const coco_tensor* out, void* stream) {
  return fused_allreduce_impl(partials, bias, residual, dropout_p, seed, 0, out, stream);
}

COCO_EXPORT coco_status coco_fused_allreduce_at(const coco_tensor* partials, const void* bias,
                                                const coco_tensor* residual, float dropout_p, uint64_t seed,
                                                uint64_t index_base, const coco_tensor* out, void* stream) {
  return fused_allreduce_impl(partials, bias, residual, dropout_p, seed, index_base, out, stream);
}

COCO_EXPORT coco_status coco_allreduce(const coco_tensor* in, const coco_tensor* out, void* stream) {
  return coco_fused_allreduce(in, nullptr, nullptr, 0.0f, 0, out, stream);
}

namespace {

// [outer, mid, inner] view of a per-rank-shaped tensor around `dim`.
void split3(const int64_t* shape, int ndim, int dim, int64_t* outer, int64_t* mid, int64_t* inner) {
  *outer = 1;
  *inner = 1;
  for (int d = 0; d < dim; ++d) *outer *= shape[d];
  *mid = shape[dim];
  for (int d = dim + 1; d < ndim; ++d) *inner *= shape[d];
}

coco_status prepare_rs(const TInfo& in, const TInfo& out, SliceLaunch* L) {
  if (in.layout != COCO_LOCAL || out.layout != COCO_SLICED) return COCO_ERR_LAYOUT;
  if (in.dtype != out.dtype) return COCO_ERR_DTYPE;
  if (!same_ranks(in, out) || in.ndim != out.ndim) return COCO_ERR_SHAPE;
  for (int d = 0; d < in.ndim; ++d)
    if (in.local[d] != out.shape[d]) return COCO_ERR_SHAPE;
  std::memset(L, 0, sizeof(*L));
  for (int i = 0; i < in.nranks * in.ngroups; ++i) {
    L->t.in[i] = in.t->ptr[i];
    L->t.out[i] = out.t->ptr[i];
  }
  L->dtype = in.dtype;
  L->nranks = in.nranks;
  L->ngroups = in.ngroups;
  split3(out.shape, out.ndim, out.slice_dim, &L->outer, &L->mid, &L->inner);
  return COCO_OK;
}

coco_status prepare_ag(const TInfo& in, const TInfo& out, SliceLaunch* L) {
  if (in.layout != COCO_SLICED || out.layout != COCO_REPLICATED) return COCO_ERR_LAYOUT;
  if (in.dtype != out.dtype) return COCO_ERR_DTYPE;
  if (!same_ranks(in, out) || in.ndim != out.ndim) return COCO_ERR_SHAPE;
  for (int d = 0; d < in.ndim; ++d)
    if (in.shape[d] != out.local[d]) return COCO_ERR_SHAPE;
  std::memset(L, 0, sizeof(*L));
  for (int i = 0; i < in.nranks * in.ngroups; ++i) L->t.in[i] = in.t->ptr[i];
  fill_outputs(out, &L->t);
  L->dtype = in.dtype;
  L->nranks = in.nranks;
  L->ngroups = in.ngroups;
  split3(in.shape, in.ndim, in.slice_dim, &L->outer, &L->mid, &L->inner);
  return COCO_OK;
}

}  // namespace

COCO_EXPORT coco_status coco_reduce_scatter(const coco_tensor* in, const coco_tensor* out, void* stream) {
  TInfo a, o;
  coco_status st;
  if ((st = check_tensor(in, &a)) != COCO_OK) return st;
  if ((st = check_tensor(out, &o)) != COCO_OK) return st;
  SliceLaunch L;
  if ((st = prepare_rs(a, o, &L)) != COCO_OK) return st;
  if (a.numel == 0) return COCO_OK;
  std::vector<Range> outs, ins;
  tensor_ranges(o, &outs);
  tensor_ranges(a, &ins);
  if ((st = check_alias(outs, ins, false)) != COCO_OK) return st;
  return cuda_status(launch_reduce_scatter(L, static_cast<cudaStream_t>(stream)));
}

COCO_EXPORT coco_status coco_allgather(const coco_tensor* in, const coco_tensor* out, void* stream) {
  TInfo a, o;
  coco_status st;
  if ((st = check_tensor(in, &a)) != COCO_OK) return st;
  if ((st = check_tensor(out, &o)) != COCO_OK) return st;
  SliceLaunch L;
  if ((st = prepare_ag(a, o, &L)) != COCO_OK) return st;
  if (o.numel == 0) return COCO_OK;
  std::vector<Range> outs, ins;
  tensor_ranges(o, &outs);
  tensor_ranges(a, &ins);
  if ((st = check_alias(outs, ins, false)) != COCO_OK) return st;
  return cuda_status(launch_allgather(L, static_cast<cudaStream_t>(stream)));
}

COCO_EXPORT coco_status coco_allreduce_rs_ag(const coco_tensor* in, const coco_tensor* scratch,
                                             const coco_tensor* out, void* stream) {
  TInfo a, sc, o;
  coco_status st;
  if ((st = check_tensor(in, &a)) != COCO_OK) return st;
  if ((st = check_tensor(scratch, &sc)) != COCO_OK) return st;
  if ((st = check_tensor(out, &o)) != COCO_OK) return st;
  SliceLaunch rs, ag;
  if ((st = prepare_rs(a, sc, &rs)) != COCO_OK) return st;
  if ((st = prepare_ag(sc, o, &ag)) != COCO_OK) return st;
  if (a.numel == 0) return COCO_OK;
  std::vector<Range> outs, ins, scr;
  tensor_ranges(o, &outs);
  tensor_ranges(a, &ins);
  tensor_ranges(sc, &scr);
  if ((st = check_alias(scr, ins, false)) != COCO_OK) return st;
  if ((st = check_alias(outs, scr, false)) != COCO_OK) return st;
  if ((st = check_alias(outs, ins, true)) != COCO_OK) return st;  // in place is safe: RS finishes first
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = cuda_status(launch_reduce_scatter(rs, s))) != COCO_OK) return st;
  return cuda_status(launch_allgather(ag, s));
}

// ------------------------------------------------------- scattered tensors

namespace {
constexpr uint32_t kScatterMagic = 0x5343544Bu;  // table header tag
constexpr int kScatterHeaderBytes = 64;

int64_t scatter_buckets(int32_t ntensors, const int64_t* numels) {
  int64_t nb = 0;
  for (int32_t t = 0; t < ntensors; ++t) nb += (numels[t] + 1023) / 1024;
  return nb;
}
}  // namespace

COCO_EXPORT size_t coco_scattered_table_bytes(int32_t ntensors, const int64_t* numels, int32_t nranks) {
  if (ntensors < 0 || nranks < 1 || (ntensors > 0 && !numels)) return 0;
  for (int32_t t = 0; t < ntensors; ++t)
    if (numels[t] < 0) return 0;
  return static_cast<size_t>(kScatterHeaderBytes) +
         static_cast<size_t>(12) * static_cast<size_t>(scatter_buckets(ntensors, numels)) * nranks;
}

COCO_EXPORT coco_status coco_scattered_table_build(int32_t ntensors, const int64_t* numels, int32_t dtype,
                                                   int32_t nranks, void* const* tensors, void* table,
                                                   size_t table_bytes, coco_scattered_plan* plan, void* stream) {
  if (!plan) return COCO_ERR_NULL;
  if (ntensors < 0 || nranks < 1 || nranks > COCO_MAX_PTRS) return COCO_ERR_SHAPE;
  if (ntensors > 0 && (!numels || !tensors)) return COCO_ERR_NULL;
  if (dtype < COCO_F32 || dtype > COCO_BF16) return COCO_ERR_DTYPE;
  for (int32_t t = 0; t < ntensors; ++t)
    if (numels[t] < 0 || numels[t] >= (int64_t(1) << 32)) return COCO_ERR_SHAPE;
  const int64_t nb = scatter_buckets(ntensors, numels);
  const size_t need = coco_scattered_table_bytes(ntensors, numels, nranks);
  if (!table) return COCO_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(table) & 15) return COCO_ERR_ALIGN;
  if (table_bytes < need) return COCO_ERR_SHAPE;
  const int es = dtype_size(dtype);
  std::vector<Range> ranges;
  for (int32_t r = 0; r < nranks; ++r)
    for (int32_t t = 0; t < ntensors; ++t) {
      if (numels[t] == 0) continue;
      const void* p = tensors[static_cast<size_t>(r) * ntensors + t];
      if (!p) return COCO_ERR_NULL;
      if (reinterpret_cast<uintptr_t>(p) & 15) return COCO_ERR_ALIGN;
      ranges.push_back(range_of(p, numels[t] * es));
    }
  ranges.push_back(range_of(table, static_cast<int64_t>(need)));
  std::sort(ranges.begin(), ranges.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < ranges.size(); ++i)
    if (ranges[i].lo < ranges[i - 1].hi) return COCO_ERR_ALIAS;

  std::vector<uint32_t> words(need / 4, 0u);
  words[0] = kScatterMagic;
  words[1] = static_cast<uint32_t>(nb & 0xFFFFFFFFu);
  words[2] = static_cast<uint32_t>(nb >> 32);
  words[3] = static_cast<uint32_t>(nranks);
  words[4] = static_cast<uint32_t>(dtype);
  words[5] = static_cast<uint32_t>(ntensors);
  size_t w = kScatterHeaderBytes / 4;
  for (int32_t t = 0; t < ntensors; ++t) {
    for (int64_t off = 0, bi = 0; off < numels[t]; off += 1024, ++bi) {
      const int64_t len = std::min<int64_t>(1024, numels[t] - off);
      const uint32_t code = static_cast<uint32_t>(bi << 10) | static_cast<uint32_t>(len - 1);
      for (int32_t r = 0; r < nranks; ++r) {
        const uint64_t a = reinterpret_cast<uint64_t>(tensors[static_cast<size_t>(r) * ntensors + t]);
        words[w++] = static_cast<uint32_t>(a & 0xFFFFFFFFu);
        words[w++] = static_cast<uint32_t>(a >> 32);
        words[w++] = code;
      }
    }
  }
  // The upload reads a temporary host buffer: a stream capture would record a copy from memory
  // freed on return, so a table is built outside capture.
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capturing) != cudaSuccess ||
      capturing != cudaStreamCaptureStatusNone) {
    (void)cudaGetLastError();
    return COCO_ERR_UNSUPPORTED;
  }
  plan->table = table;
  plan->nbuckets = nb;
  plan->nranks = nranks;
  plan->dtype = dtype;
  // pageable source: the runtime stages it before returning, so `words` may go out of scope
  return cuda_status(cudaMemcpyAsync(table, words.data(), need, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)));
}

COCO_EXPORT coco_status coco_scattered_allreduce(const coco_scattered_plan* plan, float alpha, void* stream) {
  if (!plan) return COCO_ERR_NULL;
  if (plan->nbuckets < 0 || plan->nranks < 1 || plan->nranks > COCO_MAX_PTRS) return COCO_ERR_SHAPE;
  if (plan->dtype < COCO_F32 || plan->dtype > COCO_BF16) return COCO_ERR_DTYPE;
  if (!(alpha == alpha)) return COCO_ERR_VALUE;
  if (plan->nbuckets == 0) return COCO_OK;
  if (!plan->table) return COCO_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(plan->table) & 15) return COCO_ERR_ALIGN;
  return cuda_status(launch_scattered_allreduce(plan->table, plan->nbuckets, plan->nranks, plan->dtype, alpha,
                                                static_cast<cudaStream_t>(stream)));
}

COCO_EXPORT coco_status coco_dropout_keep_mask(uint64_t seed, float dropout_p, uint64_t first_index, uint64_t count,
                                               uint8_t* mask, void* stream) {
  if (!(dropout_p >= 0.0f && dropout_p <= 1.0f)) return COCO_ERR_VALUE;
  if (count == 0) return COCO_OK;
  if (!mask) return COCO_ERR_NULL;
  const double keep = 1.0 - static_cast<double>(dropout_p);
  const uint32_t threshold = static_cast<uint32_t>(std::floor(keep * 16777216.0));
  return cuda_status(launch_keep_mask(seed, threshold, first_index, count, mask, static_cast<cudaStream_t>(stream)));
}

COCO_EXPORT coco_status coco_wait_selftest(uint64_t timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return COCO_ERR_VALUE;
  unsigned int* err = gemm_error_word();
  if (!err) return cuda_status(cudaErrorSymbolNotFound);
  return cuda_status(launch_wait_selftest(timeout_ns, static_cast<cudaStream_t>(stream), err));
}

COCO_EXPORT coco_status coco_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  unsigned int* w = gemm_error_word();
  if (!w) return cuda_status(cudaErrorSymbolNotFound);
  unsigned int v = 0;
  if ((e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_status(e);
  if (v == 0) return COCO_OK;
  if ((e = cudaMemset(w, 0, sizeof(v))) != cudaSuccess) return cuda_status(e);
  return static_cast<coco_status>(v);
}

// ------------------------------------------------------------------ einsums

namespace {

struct EinsumArgs {
  Spec spec;
  TInfo lhs, rhs, out;
};

coco_status check_einsum_common(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                const coco_tensor* out, EinsumArgs* E) {
  if (!parse_spec(spec, &E->spec)) return COCO_ERR_UNSUPPORTED;
  coco_status st;
  if ((st = check_tensor(lhs, &E->lhs)) != COCO_OK) return st;
  if ((st = check_tensor(rhs, &E->rhs)) != COCO_OK) return st;
  if ((st = check_tensor(out, &E->out)) != COCO_OK) return st;
  const int nd = E->spec.batched ? 3 : 2;
  if (E->lhs.ndim != nd || E->rhs.ndim != nd || E->out.ndim != nd) return COCO_ERR_SHAPE;
  if (E->lhs.dtype != E->rhs.dtype) return COCO_ERR_DTYPE;
  if (!same_ranks(E->lhs, E->rhs) || !same_ranks(E->lhs, E->out)) return COCO_ERR_SHAPE;
  for (int d = 0; d < nd; ++d)
    if (!fits_i32(E->lhs.shape[d]) || !fits_i32(E->rhs.shape[d]) || !fits_i32(E->out.shape[d]))
      return COCO_ERR_UNSUPPORTED;
  return COCO_OK;
}

// The pointer rank r of group g reads for a non-looped operand.
const void* operand_ptr(const TInfo& t, int g, int r) {
  return t.layout == COCO_REPLICATED ? t.ptr(g, 0) : t.ptr(g, r);
}

coco_status finish(GemmPlan& P, const EinsumArgs& E, int64_t k_total, const PlanKey& key, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (E.out.numel == 0) return COCO_OK;
  coco_status st;
  if ((st = einsum_alias(E.lhs, E.rhs, E.out)) != COCO_OK) return st;
  if (k_total == 0) return zero_outputs(E.out, s);
  P.in_dtype = E.lhs.dtype;
  P.out_dtype = E.out.dtype;
  return run_keyed(std::move(P), key, s);
}

// The cached plan of a call with these arguments, run; false if there is none.
bool run_cached(const PlanKey& key, void* stream, coco_status* st) {
  if (!key.ok) return false;
  std::shared_ptr<PlanEntry> e = plan_cache().find(key.w);
  if (!e) return false;
  *st = run_entry(*e, static_cast<cudaStream_t>(stream));
  return true;
}

}  // namespace

COCO_EXPORT coco_status coco_einsum(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                    const coco_tensor* out, void* stream) {
  PlanKey key(1);
  key.str(spec);
  key.tensor(lhs);
  key.tensor(rhs);
  key.tensor(out);
  coco_status cst;
  if (run_cached(key, stream, &cst)) return cst;
  EinsumArgs E;
  coco_status st = check_einsum_common(spec, lhs, rhs, out, &E);
  if (st != COCO_OK) return st;
  const Spec& S = E.spec;
  const int kl = S.batched ? 2 : 1, kr = S.batched ? 1 : 0;
  if (E.lhs.layout == COCO_REPLICATED) return COCO_ERR_LAYOUT;
  if (E.lhs.layout == COCO_SLICED && E.lhs.slice_dim != kl) return COCO_ERR_LAYOUT;
  if (E.rhs.layout == COCO_SLICED && E.rhs.slice_dim != kr) return COCO_ERR_LAYOUT;
  if (E.out.layout != COCO_LOCAL) return COCO_ERR_LAYOUT;
  const Dims3 a = dims_of(S, E.lhs.local), b = dims_of(S, E.rhs.local), o = dims_of(S, E.out.local);
  if (a.c != b.r || a.b != b.b || o.b != a.b || o.r != a.r || o.c != b.c) return COCO_ERR_SHAPE;
  GemmPlan P;
  for (int g = 0; g < E.out.ngroups; ++g)
    for (int r = 0; r < E.out.nranks; ++r) {
      Job J = make_job(add_out(&P, make_out(E.out.ptr(g, r), o)), o);
      J.seg0 = static_cast<int16_t>(P.segs.size());
      J.nseg = 1;
      P.segs.push_back(make_seg(add_view(&P, make_view(E.lhs.ptr(g, r), a)),
                                add_view(&P, make_view(operand_ptr(E.rhs, g, r), b)), a.c));
      P.jobs.push_back(J);
    }
  return finish(P, E, a.c, key, stream);
}

COCO_EXPORT coco_status coco_einsum_accumulate(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                               const coco_tensor* out, void* stream) {
  PlanKey key(5);
  key.str(spec);
  key.tensor(lhs);
  key.tensor(rhs);
  key.tensor(out);
  coco_status cst;
  if (run_cached(key, stream, &cst)) return cst;
  EinsumArgs E;
  coco_status st = check_einsum_common(spec, lhs, rhs, out, &E);
  if (st != COCO_OK) return st;
  const Spec& S = E.spec;
  const int kl = S.batched ? 2 : 1, kr = S.batched ? 1 : 0;
  if (E.lhs.layout == COCO_REPLICATED) return COCO_ERR_LAYOUT;
  if (E.lhs.layout == COCO_SLICED && E.lhs.slice_dim != kl) return COCO_ERR_LAYOUT;
  if (E.rhs.layout == COCO_SLICED && E.rhs.slice_dim != kr) return COCO_ERR_LAYOUT;
  if (E.out.layout != COCO_LOCAL) return COCO_ERR_LAYOUT;
  if (E.out.dtype != COCO_F32) return COCO_ERR_DTYPE;
  const Dims3 a = dims_of(S, E.lhs.local), b = dims_of(S, E.rhs.local), o = dims_of(S, E.out.local);
  if (a.c != b.r || a.b != b.b || o.b != a.b || o.r != a.r || o.c != b.c) return COCO_ERR_SHAPE;
  if (E.out.numel == 0) return COCO_OK;
  if ((st = einsum_alias(E.lhs, E.rhs, E.out)) != COCO_OK) return st;
  if (a.c == 0) return COCO_OK;  // adds nothing
  GemmPlan P;
  P.mode = EPI_ADD;
  P.in_dtype = E.lhs.dtype;
  P.out_dtype = COCO_F32;
  for (int g = 0; g < E.out.ngroups; ++g)
    for (int r = 0; r < E.out.nranks; ++r) {
      Job J = make_job(add_out(&P, make_out(E.out.ptr(g, r), o)), o);
      J.res = E.out.ptr(g, r);  // the addend is the output itself, read before it is written
      J.seg0 = static_cast<int16_t>(P.segs.size());
      J.nseg = 1;
      P.segs.push_back(make_seg(add_view(&P, make_view(E.lhs.ptr(g, r), a)),
                                add_view(&P, make_view(operand_ptr(E.rhs, g, r), b)), a.c));
      P.jobs.push_back(J);
    }
  return run_keyed(std::move(P), key, static_cast<cudaStream_t>(stream));
}

COCO_EXPORT coco_status coco_matmul_fused_allreduce(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                                    const void* bias, const coco_tensor* residual, float dropout_p,
                                                    uint64_t seed, const coco_tensor* out, void* stream) {
  PlanKey key(2);
  key.str(spec);
  key.tensor(lhs);
  key.tensor(rhs);
  key.add(reinterpret_cast<uintptr_t>(bias));
  key.tensor(residual);
  key.f32(dropout_p);
  key.add(seed);
  key.tensor(out);
  coco_status cst;
  if (run_cached(key, stream, &cst)) return cst;
  EinsumArgs E;
  coco_status st = check_einsum_common(spec, lhs, rhs, out, &E);
  if (st != COCO_OK) return st;
  if (E.spec.batched) return COCO_ERR_UNSUPPORTED;
  if (E.lhs.layout != COCO_SLICED || E.lhs.slice_dim != 1) return COCO_ERR_LAYOUT;
  if (E.rhs.layout != COCO_SLICED || E.rhs.slice_dim != 0) return COCO_ERR_LAYOUT;
  if (E.out.layout != COCO_REPLICATED) return COCO_ERR_LAYOUT;
  if (E.lhs.dtype == COCO_F32 || E.out.dtype == COCO_F32) return COCO_ERR_UNSUPPORTED;
  const Dims3 a = dims_of(E.spec, E.lhs.local), b = dims_of(E.spec, E.rhs.local), o = dims_of(E.spec, E.out.local);
  if (a.c != b.r || o.r != a.r || o.c != b.c) return COCO_ERR_SHAPE;
  TInfo res;
  if (residual) {
    if ((st = check_tensor(residual, &res)) != COCO_OK) return st;
    if (res.layout != COCO_REPLICATED) return COCO_ERR_LAYOUT;
    if (res.dtype != E.out.dtype) return COCO_ERR_DTYPE;
    if (!same_ranks(res, E.out) || !same_local_shape(res, E.out)) return COCO_ERR_SHAPE;
  }
  if (!(dropout_p >= 0.0f && dropout_p <= 1.0f)) return COCO_ERR_VALUE;
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 15)) return COCO_ERR_ALIGN;
  if (E.out.numel == 0) return COCO_OK;
  if (a.c == 0) return COCO_ERR_UNSUPPORTED;  // no contraction: use coco_fused_allreduce on zero partials
  // outputs: disjoint from the operands and bias; the residual may be an output exactly (each
  // element's residual is read by the thread that computes it, before the tile is stored)
  std::vector<Range> outs, ins, resr;
  tensor_ranges(E.out, &outs);
  tensor_ranges(E.lhs, &ins);
  tensor_ranges(E.rhs, &ins);
  if ((st = check_alias(outs, ins, false)) != COCO_OK) return st;
  if (residual) {
    tensor_ranges(res, &resr, true);
    if ((st = check_alias(outs, resr, true)) != COCO_OK) return st;
  }
  if (bias) {
    const Range br = range_of(bias, o.c * dtype_size(E.out.dtype));
    for (const Range& r : outs)
      if (overlap(r, br)) return COCO_ERR_ALIAS;
  }
  {  // a replica buffer belongs to one group only
    std::set<void*> seen;
    for (int g = 0; g < E.out.ngroups; ++g) {
      std::set<void*> mine;
      for (int r = 0; r < E.out.nranks; ++r) mine.insert(E.out.ptr(g, r));
      for (void* p : mine)
        if (!seen.insert(p).second) return COCO_ERR_ALIAS;
    }
  }

  GemmPlan P;
  P.mode = EPI_FUSED_ALLREDUCE;
  P.in_dtype = E.lhs.dtype;
  P.out_dtype = E.out.dtype;
  P.far.bias = bias;
  P.far.dropout = dropout_p > 0.0f;
  const double keep = 1.0 - static_cast<double>(dropout_p);
  P.far.keep_threshold = static_cast<uint32_t>(std::floor(keep * 16777216.0));
  P.far.scale = dropout_p < 1.0f ? static_cast<float>(1.0 / keep) : 0.0f;
  P.far.seed = seed;
  const int n = E.lhs.nranks;
  for (int g = 0; g < E.out.ngroups; ++g) {
    Job J = make_job(static_cast<int>(P.outs.size()), o);
    std::vector<int> reps = output_ranks(E.out, g);
    for (int r : reps) P.outs.push_back(make_out(E.out.ptr(g, r), o));
    J.nout = static_cast<int16_t>(reps.size());
    J.res = residual ? res.ptr(g, 0) : nullptr;
    J.seg0 = static_cast<int16_t>(P.segs.size());
    J.nseg = static_cast<int16_t>(n);
    for (int r = 0; r < n; ++r)  // the AllReduce's summation order: rank 0, 1, ..., N-1
      P.segs.push_back(make_seg(add_view(&P, make_view(E.lhs.ptr(g, r), a)),
                                add_view(&P, make_view(E.rhs.ptr(g, r), b)), a.c));
    P.jobs.push_back(J);
  }
  return run_keyed(std::move(P), key, static_cast<cudaStream_t>(stream));
}

namespace {

// The order in which rank r of n visits the shards of the looped operand.
//   ring / unroll-by-2: r, r+1, ..., r-1 (the shard held after i permutes {j -> j-1});
//   bidirectional: r, then r+1, r-1, r+2, r-2, ... (one shard from each direction per step).
std::vector<int> ag_order(int r, int n, int sched) {
  std::vector<int> o;
  if (sched != COCO_SCHED_BIDIRECTIONAL) {
    for (int i = 0; i < n; ++i) o.push_back((r + i) % n);
    return o;
  }
  o.push_back(r);
  for (int k = 1; static_cast<int>(o.size()) < n; ++k) {
    o.push_back((r + k) % n);
    if (static_cast<int>(o.size()) < n) o.push_back(((r - k) % n + n) % n);
  }
  return o;
}

// The order in which output shard r of n collects the ranks' partials.
//   ring: r-1, r-2, ..., r (the accumulator travels {j -> j-1});
//   unroll-by-2: chain r-1, r-3, ... then chain r-2, r-4, ... (two hops per iteration);
//   bidirectional: r+a, ..., r+1 (left-moving), r-b, ..., r-1 (right-moving), then r itself,
//   a = floor(n/2), b = floor((n-1)/2).
std::vector<int> rs_order(int r, int n, int sched) {
  auto md = [n](int v) { return ((v % n) + n) % n; };
  std::vector<int> o;
  if (sched == COCO_SCHED_RING) {
    for (int i = 0; i < n; ++i) o.push_back(md(r - 1 - i));
  } else if (sched == COCO_SCHED_UNROLL2) {
    for (int i = 0; i < (n + 1) / 2; ++i) o.push_back(md(r - 1 - 2 * i));
    for (int i = 0; i < n / 2; ++i) o.push_back(md(r - 2 - 2 * i));
  } else {
    const int a = n / 2, b = (n - 1) / 2;
    for (int i = 0; i < a; ++i) o.push_back(md(r + a - i));
    for (int i = 0; i < b; ++i) o.push_back(md(r - b + i));
    o.push_back(r);
  }
  return o;
}

bool valid_schedule(int sched) { return sched >= COCO_SCHED_RING && sched <= COCO_SCHED_BIDIRECTIONAL; }

coco_status looped_ag_einsum(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs, const coco_tensor* out,
                             int sched, void* stream) {
  if (!valid_schedule(sched)) return COCO_ERR_VALUE;
  PlanKey key(3);
  key.add(static_cast<uint64_t>(sched));
  key.str(spec);
  key.tensor(lhs);
  key.tensor(rhs);
  key.tensor(out);
  coco_status cst;
  if (run_cached(key, stream, &cst)) return cst;
  EinsumArgs E;
  coco_status st = check_einsum_common(spec, lhs, rhs, out, &E);
  if (st != COCO_OK) return st;
  const Spec& S = E.spec;
  const bool lhs_looped = E.lhs.layout == COCO_SLICED;
  if (lhs_looped == (E.rhs.layout == COCO_SLICED)) return COCO_ERR_LAYOUT;  // exactly one looped operand
  const TInfo& Lp = lhs_looped ? E.lhs : E.rhs;  // looped
  const TInfo& Ot = lhs_looped ? E.rhs : E.lhs;  // local operand
  if (Ot.layout == COCO_SLICED) return COCO_ERR_LAYOUT;
  if (E.out.layout == COCO_SLICED) return COCO_ERR_LAYOUT;
  if (E.out.layout == COCO_REPLICATED && Ot.layout != COCO_REPLICATED) return COCO_ERR_LAYOUT;
  const int n = Lp.nranks;
  const char lab = label(S, lhs_looped, Lp.slice_dim);

  // Full (gathered) looped operand and per-rank local operand, as [b, rows, cols].
  const Dims3 full = dims_of(S, Lp.shape), shard = dims_of(S, Lp.local), loc = dims_of(S, Ot.local);
  const Dims3 A = lhs_looped ? full : loc;  // gathered lhs
  const Dims3 B = lhs_looped ? loc : full;  // gathered rhs
  if (A.c != B.r || A.b != B.b) return COCO_ERR_SHAPE;
  const Dims3 res{A.b, A.r, B.c};
  const Dims3 o = dims_of(S, E.out.local);
  if (o.b != res.b || o.r != res.r || o.c != res.c) return COCO_ERR_SHAPE;

  GemmPlan P;
  for (int g = 0; g < Lp.ngroups; ++g) {
    for (int r : output_ranks(E.out, g)) {
      const int oi = add_out(&P, make_out(E.out.ptr(g, r), o));
      const void* other = operand_ptr(Ot, g, r);
      const std::vector<int> order = ag_order(r, n, sched);
      if (lab == 'k') {
        // case 2: one job, N K-segments in schedule order, Addition in TMEM.
        Job J = make_job(oi, res);
        J.seg0 = static_cast<int16_t>(P.segs.size());
        J.nseg = static_cast<int16_t>(n);
        const int64_t ks = lhs_looped ? shard.c : shard.r;
        for (int i = 0; i < n; ++i) {
          const int s = order[i];
          const void* sp = Lp.ptr(g, s);
          int va, vb;
          if (lhs_looped) {  // DynamicSlice rows [s*ks, (s+1)*ks) of the local rhs
            View bv = make_view(static_cast<const char*>(other) + s * ks * loc.c * dtype_size(Ot.dtype),
                                Dims3{loc.b, ks, loc.c});
            bv.bstride = loc.r * loc.c;
            va = add_view(&P, make_view(sp, shard));
            vb = add_view(&P, bv);
          } else {  // DynamicSlice columns [s*ks, (s+1)*ks) of the local lhs
            View av = make_view(static_cast<const char*>(other) + s * ks * dtype_size(Ot.dtype),
                                Dims3{loc.b, loc.r, ks});
            av.ld = loc.c;
            av.bstride = loc.r * loc.c;
            va = add_view(&P, av);
            vb = add_view(&P, make_view(sp, shard));
          }
          P.segs.push_back(make_seg(va, vb, ks));
        }
        P.jobs.push_back(J);
      } else {
        // cases 1 and 3: one job per step, DynamicUpdateSlice of shard s.
        for (int i = 0; i < n; ++i) {
          const int s = order[i];
          const void* sp = Lp.ptr(g, s);
          Dims3 ext = res;
          Job J = make_job(oi, ext);
          Seg sg;
          if (lab == 'b') {
            J.nb = static_cast<int32_t>(shard.b);
            J.o_b0 = static_cast<int32_t>(s * shard.b);
            if (lhs_looped) {
              sg = make_seg(add_view(&P, make_view(sp, shard)), add_view(&P, make_view(other, loc)), shard.c);
              sg.b_b0 = static_cast<int32_t>(s * shard.b);
            } else {
              sg = make_seg(add_view(&P, make_view(other, loc)), add_view(&P, make_view(sp, shard)), loc.c);
              sg.a_b0 = static_cast<int32_t>(s * shard.b);
            }
          } else if (lab == 'm') {  // lhs sliced on its rows
            J.m = static_cast<int32_t>(shard.r);
            J.o_r0 = static_cast<int32_t>(s * shard.r);
            sg = make_seg(add_view(&P, make_view(sp, shard)), add_view(&P, make_view(other, loc)), shard.c);
          } else {  // 'n': rhs sliced on its columns
            J.n = static_cast<int32_t>(shard.c);
            J.o_c0 = static_cast<int32_t>(s * shard.c);
            sg = make_seg(add_view(&P, make_view(other, loc)), add_view(&P, make_view(sp, shard)), loc.c);
          }
          J.seg0 = static_cast<int16_t>(P.segs.size());
          J.nseg = 1;
          P.segs.push_back(sg);
          P.jobs.push_back(J);
        }
      }
    }
  }
  return finish(P, E, A.c, key, stream);
}

coco_status looped_einsum_rs(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs, const coco_tensor* out,
                             int sched, void* stream) {
  if (!valid_schedule(sched)) return COCO_ERR_VALUE;
  PlanKey key(4);
  key.add(static_cast<uint64_t>(sched));
  key.str(spec);
  key.tensor(lhs);
  key.tensor(rhs);
  key.tensor(out);
  coco_status cst;
  if (run_cached(key, stream, &cst)) return cst;
  EinsumArgs E;
  coco_status st = check_einsum_common(spec, lhs, rhs, out, &E);
  if (st != COCO_OK) return st;
  const Spec& S = E.spec;
  const int kl = S.batched ? 2 : 1, kr = S.batched ? 1 : 0;
  if (E.lhs.layout != COCO_SLICED || E.lhs.slice_dim != kl) return COCO_ERR_LAYOUT;
  if (E.rhs.layout != COCO_SLICED || E.rhs.slice_dim != kr) return COCO_ERR_LAYOUT;
  if (E.out.layout != COCO_SLICED) return COCO_ERR_LAYOUT;
  const char olab = label(S, true, E.out.slice_dim) == 'k' ? 'n' : label(S, true, E.out.slice_dim);
  if (olab != 'm' && olab != 'n') return COCO_ERR_LAYOUT;  // partitioned on a batch dimension
  const int n = E.lhs.nranks;
  const Dims3 a = dims_of(S, E.lhs.local), b = dims_of(S, E.rhs.local);
  if (a.c != b.r || a.b != b.b) return COCO_ERR_SHAPE;
  const Dims3 og = dims_of(S, E.out.shape), ol = dims_of(S, E.out.local);
  if (og.b != a.b || og.r != a.r || og.c != b.c) return COCO_ERR_SHAPE;

  GemmPlan P;
  for (int g = 0; g < E.out.ngroups; ++g) {
    for (int r = 0; r < n; ++r) {
      Job J = make_job(add_out(&P, make_out(E.out.ptr(g, r), ol)), ol);
      J.seg0 = static_cast<int16_t>(P.segs.size());
      J.nseg = static_cast<int16_t>(n);
      const std::vector<int> order = rs_order(r, n, sched);
      for (int i = 0; i < n; ++i) {
        const int q = order[i];  // the order in which the accumulated shard r collects partials
        Seg sg = make_seg(add_view(&P, make_view(E.lhs.ptr(g, q), a)), add_view(&P, make_view(E.rhs.ptr(g, q), b)),
                          a.c);
        if (olab == 'm') sg.a_r0 = static_cast<int32_t>(r * ol.r);  // DynamicSlice of lhs rows
        else sg.b_c0 = static_cast<int32_t>(r * ol.c);              // DynamicSlice of rhs columns
        P.segs.push_back(sg);
      }
      P.jobs.push_back(J);
    }
  }
  return finish(P, E, a.c, key, stream);
}

}  // namespace

COCO_EXPORT coco_status coco_looped_ag_einsum(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                              const coco_tensor* out, void* stream) {
  return looped_ag_einsum(spec, lhs, rhs, out, COCO_SCHED_RING, stream);
}

COCO_EXPORT coco_status coco_looped_ag_einsum_sched(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                                    const coco_tensor* out, int schedule, void* stream) {
  return looped_ag_einsum(spec, lhs, rhs, out, schedule, stream);
}

COCO_EXPORT coco_status coco_looped_einsum_rs(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                              const coco_tensor* out, void* stream) {
  return looped_einsum_rs(spec, lhs, rhs, out, COCO_SCHED_RING, stream);
}

COCO_EXPORT coco_status coco_looped_einsum_rs_sched(const char* spec, const coco_tensor* lhs, const coco_tensor* rhs,
                                                    const coco_tensor* out, int schedule, void* stream) {
  return looped_einsum_rs(spec, lhs, rhs, out, schedule, stream);
}

COCO_EXPORT coco_status coco_shard_order(int32_t kind, int32_t schedule, int32_t rank, int32_t nranks,
                                         int32_t* order) {
  if (!order) return COCO_ERR_NULL;
  if (nranks < 1 || nranks > COCO_MAX_PTRS || rank < 0 || rank >= nranks) return COCO_ERR_SHAPE;
  if ((kind != 0 && kind != 1) || !valid_schedule(schedule)) return COCO_ERR_VALUE;
  const std::vector<int> o = kind == 0 ? ag_order(rank, nranks, schedule) : rs_order(rank, nranks, schedule);
  for (int i = 0; i < nranks; ++i) order[i] = o[i];
  return COCO_OK;
}

// [Decomp] §5.5: decompose only when
//   orig_comp + orig_comm >= max(orig_comp, ring_comm) + epilogue_cost.
COCO_EXPORT coco_status coco_loop_profitable(double orig_comp, double orig_comm, double ring_comm,
                                             double epilogue_cost, int32_t* profitable) {
  if (!profitable) return COCO_ERR_NULL;
  for (double t : {orig_comp, orig_comm, ring_comm, epilogue_cost})
    if (!std::isfinite(t) || t < 0.0) return COCO_ERR_VALUE;
  *profitable = orig_comp + orig_comm >= std::max(orig_comp, ring_comm) + epilogue_cost ? 1 : 0;
  return COCO_OK;
}

COCO_EXPORT void coco_plan_cache_stats(uint64_t* hits, uint64_t* misses, uint64_t* entries) {
  plan_cache().stats(hits, misses, entries);
}

COCO_EXPORT void coco_plan_cache_clear(void) { plan_cache().clear(); }
