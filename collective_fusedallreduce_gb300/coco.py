"""Thin Python binding of libcoco (include/coco.h): argument marshalling only.

Each ``coco_*`` function here has the name and argument order of the C entry
point. Distributed tensors are described with ``local``, ``sliced`` and
``replicated`` ([CoCoNet] "Breaking the Computation and Communication
Abstraction Barrier in Distributed Machine Learning Workloads", tensor
layouts) from per-rank ``torch.Tensor`` lists (group-major for several
groups); PyTorch provides device memory and streams, every computation runs in
the library's kernels. A failing call raises ``CocoError``.

Importing this module loads ``libcoco.so`` from this package directory and
raises ``ImportError`` if it has not been built (``__graft_entry__.build()``):
there is no fallback.
"""

import ctypes
import os

import torch

# COCO_LIBRARY selects another build of the same library (e.g. build.build_sanitized's).
_LIB_PATH = os.environ.get("COCO_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcoco.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build()")
_lib = ctypes.CDLL(_LIB_PATH)

MAX_PTRS = 64
MAX_DIMS = 3

F32, F16, BF16 = 0, 1, 2
LOCAL, SLICED, REPLICATED = 0, 1, 2
SCHED_RING, SCHED_UNROLL2, SCHED_BIDIRECTIONAL = 0, 1, 2

STATUS = {
    0: "COCO_OK", 1: "COCO_ERR_NULL", 2: "COCO_ERR_SHAPE", 3: "COCO_ERR_DTYPE", 4: "COCO_ERR_LAYOUT",
    5: "COCO_ERR_ALIGN", 6: "COCO_ERR_ALIAS", 7: "COCO_ERR_UNSUPPORTED", 8: "COCO_ERR_CUDA",
    9: "COCO_ERR_TIMEOUT", 10: "COCO_ERR_VALUE",
}

_DTYPES = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


class CocoTensor(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("slice_dim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * MAX_DIMS),
        ("nranks", ctypes.c_int32),
        ("ngroups", ctypes.c_int32),
        ("ptr", ctypes.c_void_p * MAX_PTRS),
    ]


class CocoScatteredPlan(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("nbuckets", ctypes.c_int64), ("nranks", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class CocoError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        self.name = STATUS.get(status, str(status))
        msg = _lib.coco_status_string(status).decode()
        if status == 8:
            msg += f" (cudaError {_lib.coco_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


_P = ctypes.POINTER(CocoTensor)
_S = ctypes.c_void_p
for _name, _args in {
    "coco_fused_allreduce": [_P, ctypes.c_void_p, _P, ctypes.c_float, ctypes.c_uint64, _P, _S],
    "coco_fused_allreduce_at": [_P, ctypes.c_void_p, _P, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64, _P, _S],
    "coco_allreduce": [_P, _P, _S],
    "coco_reduce_scatter": [_P, _P, _S],
    "coco_allgather": [_P, _P, _S],
    "coco_allreduce_rs_ag": [_P, _P, _P, _S],
    "coco_allreduce_rs_ag_noalloc": [_P, _P, _S],
    "coco_einsum": [ctypes.c_char_p, _P, _P, _P, _S],
    "coco_einsum_accumulate": [ctypes.c_char_p, _P, _P, _P, _S],
    "coco_matmul_fused_allreduce": [ctypes.c_char_p, _P, _P, ctypes.c_void_p, _P, ctypes.c_float, ctypes.c_uint64,
                                    _P, _S],
    "coco_looped_ag_einsum": [ctypes.c_char_p, _P, _P, _P, _S],
    "coco_looped_einsum_rs": [ctypes.c_char_p, _P, _P, _P, _S],
    "coco_looped_ag_einsum_sched": [ctypes.c_char_p, _P, _P, _P, ctypes.c_int, _S],
    "coco_looped_einsum_rs_sched": [ctypes.c_char_p, _P, _P, _P, ctypes.c_int, _S],
    "coco_dropout_keep_mask": [ctypes.c_uint64, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p, _S],
    "coco_device_status": [_S],
    "coco_wait_selftest": [ctypes.c_uint64, _S],
}.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.coco_scattered_table_bytes.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]
_lib.coco_scattered_table_bytes.restype = ctypes.c_size_t
_lib.coco_scattered_table_build.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32,
                                            ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p,
                                            ctypes.c_size_t, ctypes.POINTER(CocoScatteredPlan), _S]
_lib.coco_scattered_table_build.restype = ctypes.c_int
_lib.coco_scattered_allreduce.argtypes = [ctypes.POINTER(CocoScatteredPlan), ctypes.c_float, _S]
_lib.coco_scattered_allreduce.restype = ctypes.c_int
_lib.coco_status_string.argtypes = [ctypes.c_int]
_lib.coco_status_string.restype = ctypes.c_char_p
_lib.coco_last_cuda_error.restype = ctypes.c_int
_lib.coco_version.restype = ctypes.c_int
_lib.coco_kernel_launches.restype = ctypes.c_uint64
_lib.coco_shard_order.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.POINTER(ctypes.c_int32)]
_lib.coco_shard_order.restype = ctypes.c_int
_lib.coco_loop_profitable.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                      ctypes.POINTER(ctypes.c_int32)]
_lib.coco_loop_profitable.restype = ctypes.c_int
_lib.coco_plan_cache_stats.argtypes = [ctypes.POINTER(ctypes.c_uint64)] * 3
_lib.coco_plan_cache_stats.restype = None
_lib.coco_plan_cache_clear.argtypes = []
_lib.coco_plan_cache_clear.restype = None

EXPORTED = [
    "coco_fused_allreduce", "coco_fused_allreduce_at", "coco_allreduce", "coco_reduce_scatter", "coco_allgather", "coco_allreduce_rs_ag",
    "coco_allreduce_rs_ag_noalloc",
    "coco_einsum", "coco_einsum_accumulate", "coco_matmul_fused_allreduce", "coco_looped_ag_einsum", "coco_looped_einsum_rs",
    "coco_looped_ag_einsum_sched", "coco_looped_einsum_rs_sched", "coco_dropout_keep_mask",
    "coco_scattered_table_bytes", "coco_scattered_table_build", "coco_scattered_allreduce",
    "coco_device_status", "coco_wait_selftest", "coco_kernel_launches", "coco_last_cuda_error", "coco_status_string", "coco_version",
    "coco_shard_order", "coco_loop_profitable", "coco_plan_cache_stats", "coco_plan_cache_clear",
]


def library_path():
    return _LIB_PATH


def version():
    return _lib.coco_version()


def coco_kernel_launches():
    return int(_lib.coco_kernel_launches())


# ------------------------------------------------------------ tensor specs


class Dist:
    """A distributed tensor: per-rank tensors plus layout (marshalled to coco_tensor)."""

    def __init__(self, layout, tensors, shape, slice_dim=-1, ngroups=1, dtype=None):
        self.layout = layout
        self.tensors = list(tensors)
        self.shape = tuple(int(s) for s in shape)
        self.slice_dim = slice_dim
        self.ngroups = ngroups
        self.nranks = len(self.tensors) // ngroups
        self.dtype = dtype if dtype is not None else _DTYPES[self.tensors[0].dtype]

    def c(self):
        t = CocoTensor()
        t.dtype = self.dtype
        t.layout = self.layout
        t.ndim = len(self.shape)
        t.slice_dim = self.slice_dim
        for i, s in enumerate(self.shape):
            t.shape[i] = s
        t.nranks = self.nranks
        t.ngroups = self.ngroups
        for i, x in enumerate(self.tensors):
            t.ptr[i] = x.data_ptr() if x is not None else None
        return t


def local(tensors, ngroups=1):
    """Same shape, different values on every rank."""
    return Dist(LOCAL, tensors, tensors[0].shape, ngroups=ngroups)


def replicated(tensors, ngroups=1):
    """Same values on every rank (a single tensor may be repeated)."""
    return Dist(REPLICATED, tensors, tensors[0].shape, ngroups=ngroups)


def sliced(tensors, dim, ngroups=1):
    """Rank r holds slice r of a tensor split equally along ``dim``."""
    nranks = len(tensors) // ngroups
    shape = list(tensors[0].shape)
    shape[dim] *= nranks
    return Dist(SLICED, tensors, shape, slice_dim=dim, ngroups=ngroups)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ref(d):
    return None if d is None else ctypes.byref(d.c())


def _check(status, where):
    if status != 0:
        raise CocoError(status, where)


# ------------------------------------------------------------- entry points


def coco_fused_allreduce(partials, bias, residual, dropout_p, seed, out, stream=None):
    bias_ptr = None if bias is None else ctypes.c_void_p(bias.data_ptr())
    _check(_lib.coco_fused_allreduce(_ref(partials), bias_ptr, _ref(residual), float(dropout_p), int(seed),
                                     _ref(out), _stream(stream)), "coco_fused_allreduce")


def coco_fused_allreduce_at(partials, bias, residual, dropout_p, seed, index_base, out, stream=None):
    """coco_fused_allreduce over a contiguous part of larger tensors; index_base is the whole-tensor
    row-major index of the part's first element (dropout indices and bias phase continue from it)."""
    bias_ptr = None if bias is None else ctypes.c_void_p(bias.data_ptr())
    _check(_lib.coco_fused_allreduce_at(_ref(partials), bias_ptr, _ref(residual), float(dropout_p), int(seed),
                                        int(index_base), _ref(out), _stream(stream)), "coco_fused_allreduce_at")


def coco_allreduce(inp, out, stream=None):
    _check(_lib.coco_allreduce(_ref(inp), _ref(out), _stream(stream)), "coco_allreduce")


def coco_reduce_scatter(inp, out, stream=None):
    _check(_lib.coco_reduce_scatter(_ref(inp), _ref(out), _stream(stream)), "coco_reduce_scatter")


def coco_allgather(inp, out, stream=None):
    _check(_lib.coco_allgather(_ref(inp), _ref(out), _stream(stream)), "coco_allgather")


def coco_allreduce_rs_ag(inp, scratch, out, stream=None):
    _check(_lib.coco_allreduce_rs_ag(_ref(inp), _ref(scratch), _ref(out), _stream(stream)), "coco_allreduce_rs_ag")


def coco_allreduce_rs_ag_noalloc(inp, out, stream=None):
    """RS-AG with the library's fixed scratch array (for callers that cannot allocate)."""
    _check(_lib.coco_allreduce_rs_ag_noalloc(_ref(inp), _ref(out), _stream(stream)), "coco_allreduce_rs_ag_noalloc")


def coco_einsum(spec, lhs, rhs, out, stream=None):
    _check(_lib.coco_einsum(spec.encode(), _ref(lhs), _ref(rhs), _ref(out), _stream(stream)), "coco_einsum")


def coco_einsum_accumulate(spec, lhs, rhs, out, stream=None):
    _check(_lib.coco_einsum_accumulate(spec.encode(), _ref(lhs), _ref(rhs), _ref(out), _stream(stream)),
           "coco_einsum_accumulate")


def coco_matmul_fused_allreduce(spec, lhs, rhs, bias, residual, dropout_p, seed, out, stream=None):
    bias_ptr = None if bias is None else ctypes.c_void_p(bias.data_ptr())
    _check(_lib.coco_matmul_fused_allreduce(spec.encode(), _ref(lhs), _ref(rhs), bias_ptr, _ref(residual),
                                            float(dropout_p), int(seed), _ref(out), _stream(stream)),
           "coco_matmul_fused_allreduce")


def coco_looped_ag_einsum(spec, lhs, rhs, out, stream=None):
    _check(_lib.coco_looped_ag_einsum(spec.encode(), _ref(lhs), _ref(rhs), _ref(out), _stream(stream)),
           "coco_looped_ag_einsum")


def coco_looped_einsum_rs(spec, lhs, rhs, out, stream=None):
    _check(_lib.coco_looped_einsum_rs(spec.encode(), _ref(lhs), _ref(rhs), _ref(out), _stream(stream)),
           "coco_looped_einsum_rs")


def coco_looped_ag_einsum_sched(spec, lhs, rhs, out, schedule, stream=None):
    _check(_lib.coco_looped_ag_einsum_sched(spec.encode(), _ref(lhs), _ref(rhs), _ref(out), int(schedule),
                                            _stream(stream)), "coco_looped_ag_einsum_sched")


def coco_looped_einsum_rs_sched(spec, lhs, rhs, out, schedule, stream=None):
    _check(_lib.coco_looped_einsum_rs_sched(spec.encode(), _ref(lhs), _ref(rhs), _ref(out), int(schedule),
                                            _stream(stream)), "coco_looped_einsum_rs_sched")


def coco_dropout_keep_mask(seed, dropout_p, first_index, count, mask, stream=None):
    ptr = None if mask is None else ctypes.c_void_p(mask.data_ptr())
    _check(_lib.coco_dropout_keep_mask(int(seed), float(dropout_p), int(first_index), int(count), ptr,
                                       _stream(stream)), "coco_dropout_keep_mask")


def coco_device_status(stream=None):
    _check(_lib.coco_device_status(_stream(stream)), "coco_device_status")


def coco_wait_selftest(timeout_ns, stream=None):
    """Launches the failure-path self-test: a bounded wait on a barrier nothing completes
    (``timeout_ns`` limit); the next coco_device_status raises COCO_ERR_TIMEOUT."""
    _check(_lib.coco_wait_selftest(int(timeout_ns), _stream(stream)), "coco_wait_selftest")


def raw_call(name, *args):
    """Calls a C entry point with already-marshalled ctypes arguments and
    returns its status code (used by the interface tests)."""
    return getattr(_lib, name)(*args)


def coco_scattered_table_bytes(numels, nranks):
    arr = (ctypes.c_int64 * len(numels))(*[int(n) for n in numels])
    return int(_lib.coco_scattered_table_bytes(len(numels), arr, int(nranks)))


def coco_scattered_table_build(per_rank, table, stream=None):
    """``per_rank[r][t]``: rank r's tensor t (same sizes and dtype on every rank);
    ``table``: a device uint8 tensor of at least coco_scattered_table_bytes() bytes.
    Returns the plan for coco_scattered_allreduce."""
    nranks, ntensors = len(per_rank), len(per_rank[0])
    numels = (ctypes.c_int64 * ntensors)(*[x.numel() for x in per_rank[0]])
    ptrs = (ctypes.c_void_p * (nranks * ntensors))(*[x.data_ptr() if x.numel() else None
                                                     for row in per_rank for x in row])
    plan = CocoScatteredPlan()
    dtype = _DTYPES[per_rank[0][0].dtype] if ntensors else F32
    _check(_lib.coco_scattered_table_build(ntensors, numels, dtype, nranks, ptrs, ctypes.c_void_p(table.data_ptr()),
                                           table.numel() * table.element_size(), ctypes.byref(plan), _stream(stream)),
           "coco_scattered_table_build")
    return plan


def coco_scattered_allreduce(plan, alpha=1.0, stream=None):
    _check(_lib.coco_scattered_allreduce(ctypes.byref(plan), float(alpha), _stream(stream)), "coco_scattered_allreduce")


AG_ORDER, RS_ORDER = 0, 1


def coco_shard_order(kind, schedule, rank, nranks):
    """The planner's shard schedule for one rank (see coco.h): kind AG_ORDER gives the shard visited at
    each AllGather-Einsum step, RS_ORDER the rank whose partial output shard ``rank`` collects at each
    Einsum-ReduceScatter step."""
    arr = (ctypes.c_int32 * max(1, int(nranks)))()
    _check(_lib.coco_shard_order(int(kind), int(schedule), int(rank), int(nranks), arr), "coco_shard_order")
    return [int(arr[i]) for i in range(int(nranks))]


def coco_loop_profitable(orig_comp, orig_comm, ring_comm, epilogue_cost):
    """[Decomp] §5.5 cost model: True when the Looped CollectiveEinsum is expected to beat the original
    collective followed by the einsum (times in one unit)."""
    out = ctypes.c_int32(-1)
    _check(_lib.coco_loop_profitable(float(orig_comp), float(orig_comm), float(ring_comm), float(epilogue_cost),
                                     ctypes.byref(out)), "coco_loop_profitable")
    return bool(out.value)


def coco_plan_cache_stats():
    """(hits, misses, entries) of the library's plan cache."""
    h, m, e = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    _lib.coco_plan_cache_stats(ctypes.byref(h), ctypes.byref(m), ctypes.byref(e))
    return int(h.value), int(m.value), int(e.value)


def coco_plan_cache_clear():
    _lib.coco_plan_cache_clear()
