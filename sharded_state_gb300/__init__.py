"""Python binding of libshardstate (the GB300 sharded-state step, C ABI in
include/shardstate.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Functions keep the C names.  Tensors are passed as torch tensors (or
raw integer device addresses); torch supplies device memory and streams.

The library must have been built (``python sharded_state_gb300/build.py`` or
``__graft_entry__.build()``); importing this package raises if it is missing,
and there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libshardstate.so")

SS_OK = 0
SS_EINVAL = -1
SS_EALIGN = -2
SS_EOVERFLOW = -3
SS_ENOMEM = -4
SS_ECUDA = -5
SS_ENODEVICE = -6
SS_ESCRATCH = -7
SS_DDP_NOALLOC_TABLE_BYTES = 256 * 1024

SS_FLAT_ORIG_FALSE = 0
SS_FLAT_ORIG_TRUE = 1
SS_PER_PARAM_DIM0 = 2
SS_PLAN_HOST_ONLY = 1
SS_MAX_WORLD = 64
SS_MAX_REPLICAS = 64

# every symbol include/shardstate.h declares
EXPORTED = ("fsdp_plan_create", "fsdp_plan_layout", "fsdp_plan_info", "fsdp_plan_param_offset",
            "fsdp_plan_group", "fsdp_plan_destroy", "fsdp_pack", "fsdp_init_master",
            "fsdp_reduce_scatter_adamw", "fsdp_all_gather_unpack", "ddp_bucket_pack_average",
            "ddp_bucket_assign", "ss_strerror", "ss_last_cuda_error", "ss_version",
            "ss_launch_count", "ddp_bucket_pack_average_noalloc", "fsdp_sharded_step",
            "fsdp_reduce_scatter_accumulate", "fsdp_plan_validate")


class ShardStateError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({detail})")


class _PlanDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("world_size", ctypes.c_int), ("elem_bytes", ctypes.c_int),
                ("num_params", ctypes.c_int), ("dim0", ctypes.POINTER(ctypes.c_int64)),
                ("inner", ctypes.POINTER(ctypes.c_int64)), ("num_groups", ctypes.c_int),
                ("group_num_params", ctypes.POINTER(ctypes.c_int)), ("flags", ctypes.c_uint)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("shard_numel", ctypes.c_int64), ("total_numel", ctypes.c_int64),
                ("unpadded_numel", ctypes.c_int64), ("pad_numel", ctypes.c_int64),
                ("world_size", ctypes.c_int), ("elem_bytes", ctypes.c_int),
                ("num_params", ctypes.c_int), ("num_groups", ctypes.c_int), ("kind", ctypes.c_int),
                ("has_device_metadata", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class AdamW(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("step", ctypes.c_int64)]


class _Step(ctypes.Structure):
    _fields_ = [("rank_grads", ctypes.c_void_p), ("rank_param_grads", ctypes.c_void_p),
                ("master", ctypes.c_void_p), ("exp_avg", ctypes.c_void_p),
                ("exp_avg_sq", ctypes.c_void_p), ("param_shards", ctypes.c_void_p),
                ("hp", ctypes.POINTER(AdamW)), ("reduced_grad_out", ctypes.c_void_p),
                ("params_out", ctypes.c_void_p), ("n_out", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python sharded_state_gb300/build.py` "
                          "(nvcc, sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    i64p = ctypes.POINTER(ctypes.c_int64)
    vpp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "fsdp_plan_create": ([ctypes.POINTER(_PlanDesc), ctypes.POINTER(vp)], i32),
        "fsdp_plan_layout": ([i32, i32, i32, i32, i64p, i64p, ctypes.POINTER(vp)], i32),
        "fsdp_plan_info": ([vp, ctypes.POINTER(PlanInfo)], i32),
        "fsdp_plan_param_offset": ([vp, i32, i64p, i64p], i32),
        "fsdp_plan_group": ([vp, i32, i64p, i64p, ctypes.POINTER(i32), ctypes.POINTER(i32)], i32),
        "fsdp_plan_destroy": ([vp], None),
        "fsdp_plan_validate": ([vp], i32),
        "fsdp_pack": ([vp, vpp, vp, i32, vp], i32),
        "fsdp_init_master": ([vp, vp, vp, vp, vp, i32, vp], i32),
        "fsdp_reduce_scatter_adamw": ([vp, vpp, vp, vp, vp, vp, ctypes.POINTER(AdamW), vp, i32, vp],
                                      i32),
        "fsdp_all_gather_unpack": ([vp, vp, vpp, i32, i32, vp], i32),
        "ddp_bucket_pack_average": ([i32, i32, i64p, vpp, ctypes.c_size_t, vpp,
                                     ctypes.POINTER(i32), vp], i32),
        "ddp_bucket_pack_average_noalloc": ([i32, i32, i64p, vpp, ctypes.c_size_t, vpp,
                                             ctypes.POINTER(i32), vp], i32),
        "ddp_bucket_assign": ([i32, i64p, i32, ctypes.c_size_t, ctypes.POINTER(i32)], i32),
        "fsdp_sharded_step": ([vp, ctypes.POINTER(_Step), i32, vp], i32),
        "fsdp_reduce_scatter_accumulate": ([vp, vpp, vp, i32, i32, vp, vp, vp, vp,
                                            ctypes.POINTER(AdamW), vp, i32, vp], i32),
        "ss_strerror": ([i32], ctypes.c_char_p),
        "ss_last_cuda_error": ([], i32),
        "ss_version": ([], ctypes.c_char_p),
        "ss_launch_count": ([], ctypes.c_uint64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def ss_strerror(status: int) -> str:
    return _lib.ss_strerror(status).decode()


def ss_last_cuda_error() -> int:
    return int(_lib.ss_last_cuda_error())


def ss_version() -> str:
    return _lib.ss_version().decode()


def ss_launch_count() -> int:
    return int(_lib.ss_launch_count())


def _check(fn: str, status: int) -> None:
    if status != SS_OK:
        detail = ss_strerror(status)
        if status == SS_ECUDA:
            detail += f", cudaError {ss_last_cuda_error()}"
        raise ShardStateError(fn, status, detail)


def _addr(x) -> Optional[int]:
    """Device address of a tensor (or an int / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def ptr_array(xs: Sequence) -> ctypes.Array:
    """A host array of device pointers, built once and reusable across calls
    (every call that takes a list of tensors also accepts one of these)."""
    return _ptr_array(xs)


def _ptr_array(xs: Sequence) -> ctypes.Array:
    if isinstance(xs, ctypes.Array):
        return xs
    arr = (ctypes.c_void_p * max(1, len(xs)))()
    for k, x in enumerate(xs):
        arr[k] = _addr(x)
    return arr


def _i64_array(xs: Sequence[int]):
    arr = (ctypes.c_int64 * max(1, len(xs)))()
    for k, x in enumerate(xs):
        arr[k] = int(x)
    return arr


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


# ---------------------------------------------------------------------------
# plans
# ---------------------------------------------------------------------------

class Plan:
    """Owns an ss_plan*; destroyed with the object (or explicitly via destroy())."""

    def __init__(self, handle: int):
        self.handle = handle

    @property
    def _as_parameter_(self):
        return ctypes.c_void_p(self.handle)

    def info(self) -> PlanInfo:
        return fsdp_plan_info(self)

    def destroy(self) -> None:
        if self.handle:
            _lib.fsdp_plan_destroy(ctypes.c_void_p(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def fsdp_plan_create(kind: int, world_size: int, elem_bytes: int, dim0: Sequence[int],
                     inner: Optional[Sequence[int]] = None,
                     group_num_params: Optional[Sequence[int]] = None,
                     host_only: bool = False) -> Plan:
    n = len(dim0)
    d0 = _i64_array(dim0)
    inn = _i64_array(inner) if inner is not None else None
    groups = None
    if group_num_params is not None:
        groups = (ctypes.c_int * max(1, len(group_num_params)))(*group_num_params)
    desc = _PlanDesc(kind, world_size, elem_bytes, n,
                     ctypes.cast(d0, ctypes.POINTER(ctypes.c_int64)),
                     ctypes.cast(inn, ctypes.POINTER(ctypes.c_int64)) if inn is not None else None,
                     len(group_num_params) if group_num_params is not None else 0,
                     ctypes.cast(groups, ctypes.POINTER(ctypes.c_int)) if groups is not None else None,
                     SS_PLAN_HOST_ONLY if host_only else 0)
    out = ctypes.c_void_p()
    _check("fsdp_plan_create", _lib.fsdp_plan_create(ctypes.byref(desc), ctypes.byref(out)))
    return Plan(out.value)


def fsdp_plan_layout(kind: int, world_size: int, elem_bytes: int, dim0: Sequence[int],
                     inner: Optional[Sequence[int]] = None) -> Plan:
    d0 = _i64_array(dim0)
    inn = _i64_array(inner) if inner is not None else None
    out = ctypes.c_void_p()
    _check("fsdp_plan_layout", _lib.fsdp_plan_layout(
        kind, world_size, elem_bytes, len(dim0), ctypes.cast(d0, ctypes.POINTER(ctypes.c_int64)),
        ctypes.cast(inn, ctypes.POINTER(ctypes.c_int64)) if inn is not None else None,
        ctypes.byref(out)))
    return Plan(out.value)


def fsdp_plan_info(plan: Plan) -> PlanInfo:
    info = PlanInfo()
    _check("fsdp_plan_info", _lib.fsdp_plan_info(plan, ctypes.byref(info)))
    return info


def fsdp_plan_param_offset(plan: Plan, param: int):
    off = ctypes.c_int64()
    rows = ctypes.c_int64()
    _check("fsdp_plan_param_offset",
           _lib.fsdp_plan_param_offset(plan, param, ctypes.byref(off), ctypes.byref(rows)))
    return off.value, rows.value


def fsdp_plan_group(plan: Plan, group: int):
    base, shard = ctypes.c_int64(), ctypes.c_int64()
    first, count = ctypes.c_int(), ctypes.c_int()
    _check("fsdp_plan_group", _lib.fsdp_plan_group(plan, group, ctypes.byref(base),
                                                   ctypes.byref(shard), ctypes.byref(first),
                                                   ctypes.byref(count)))
    return {"base": base.value, "shard_numel": shard.value, "first_param": first.value,
            "num_params": count.value}


def fsdp_plan_validate(plan: Plan) -> None:
    _check("fsdp_plan_validate", _lib.fsdp_plan_validate(plan))


def fsdp_plan_destroy(plan: Plan) -> None:
    plan.destroy()


# ---------------------------------------------------------------------------
# step
# ---------------------------------------------------------------------------

def fsdp_pack(plan: Plan, params: Sequence, packed, group: int = -1, stream=None) -> None:
    _check("fsdp_pack", _lib.fsdp_pack(plan, _ptr_array(params), _addr(packed), group,
                                       _stream(stream)))


def fsdp_init_master(plan: Plan, param_shards, master, exp_avg, exp_avg_sq, group: int = -1,
                     stream=None) -> None:
    _check("fsdp_init_master", _lib.fsdp_init_master(plan, _addr(param_shards), _addr(master),
                                                     _addr(exp_avg), _addr(exp_avg_sq), group,
                                                     _stream(stream)))


def adamw_params(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1) -> AdamW:
    return AdamW(lr, beta1, beta2, eps, weight_decay, step)


def fsdp_reduce_scatter_adamw(plan: Plan, rank_grads: Sequence, master, exp_avg, exp_avg_sq,
                              param_shards, hp: Optional[AdamW], reduced_grad_out=None,
                              group: int = -1, stream=None) -> None:
    _check("fsdp_reduce_scatter_adamw", _lib.fsdp_reduce_scatter_adamw(
        plan, _ptr_array(rank_grads), _addr(master), _addr(exp_avg), _addr(exp_avg_sq),
        _addr(param_shards), ctypes.byref(hp) if hp is not None else None, _addr(reduced_grad_out),
        group, _stream(stream)))


def fsdp_reduce_scatter_accumulate(plan: Plan, rank_grads: Sequence, accum, micro_step: int,
                                   num_micro: int, master=None, exp_avg=None, exp_avg_sq=None,
                                   param_shards=None, hp: Optional[AdamW] = None,
                                   reduced_grad_out=None, group: int = -1, stream=None) -> None:
    """Micro-batch `micro_step` of `num_micro`: accumulate the reduce-scatter in
    fp32, and on the last micro-batch run AdamW on the micro-batch mean."""
    _check("fsdp_reduce_scatter_accumulate", _lib.fsdp_reduce_scatter_accumulate(
        plan, _ptr_array(rank_grads), _addr(accum), micro_step, num_micro, _addr(master),
        _addr(exp_avg), _addr(exp_avg_sq), _addr(param_shards),
        ctypes.byref(hp) if hp is not None else None, _addr(reduced_grad_out), group,
        _stream(stream)))


def fsdp_all_gather_unpack(plan: Plan, param_shards, params_out: Sequence, n_out: int = 1,
                           group: int = -1, stream=None) -> None:
    """params_out: n_out * num_params tensors, replica-major."""
    _check("fsdp_all_gather_unpack", _lib.fsdp_all_gather_unpack(
        plan, _addr(param_shards), _ptr_array(params_out), n_out, group, _stream(stream)))


def fsdp_sharded_step(plan: Plan, master, exp_avg, exp_avg_sq, param_shards, hp: AdamW,
                      rank_grads: Optional[Sequence] = None,
                      rank_param_grads: Optional[Sequence] = None, params_out=None,
                      n_out: int = 0, reduced_grad_out=None, group: int = -1,
                      stream=None) -> None:
    """One-pass step: gradients from N packed buffers (rank_grads) or from N
    per-parameter gradient sets (rank_param_grads, rank-major: rank r's
    gradient of parameter i at r*num_params + i), reduce-scatter + AdamW, and
    optionally the n_out per-parameter outputs (replica-major)."""
    keep = []
    def arr(xs):
        if xs is None:
            return None
        a = _ptr_array(xs)
        keep.append(a)
        return ctypes.cast(a, ctypes.c_void_p)
    st = _Step(arr(rank_grads), arr(rank_param_grads), _addr(master), _addr(exp_avg),
               _addr(exp_avg_sq), _addr(param_shards), ctypes.pointer(hp), _addr(reduced_grad_out),
               arr(params_out) if n_out > 0 else None, n_out)
    _check("fsdp_sharded_step", _lib.fsdp_sharded_step(plan, ctypes.byref(st), group,
                                                       _stream(stream)))


class ShardedStep:
    """fsdp_sharded_step with every argument marshalled once, for loops whose
    steps are short enough that building the call each time shows: a call
    sets the AdamW step number (the other hyper-parameters are the ones given
    here) and runs the step on `stream`, an int handle (0: the legacy default
    stream) fixed here.  Keeps the pointer arrays alive; the tensors must stay
    alive and in place as long as the object is used."""

    def __init__(self, plan: Plan, master, exp_avg, exp_avg_sq, param_shards, hp: AdamW,
                 rank_grads: Optional[Sequence] = None,
                 rank_param_grads: Optional[Sequence] = None, params_out=None, n_out: int = 0,
                 reduced_grad_out=None, group: int = -1, stream=None):
        self._plan = plan  # keeps the plan alive
        self._pp = ctypes.c_void_p(plan.handle)
        self._hp = AdamW(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step)
        self._keep = []

        def arr(xs):
            if xs is None:
                return None
            a = _ptr_array(xs)
            self._keep.append(a)
            return ctypes.cast(a, ctypes.c_void_p)
        self._st = _Step(arr(rank_grads), arr(rank_param_grads), _addr(master), _addr(exp_avg),
                         _addr(exp_avg_sq), _addr(param_shards), ctypes.pointer(self._hp),
                         _addr(reduced_grad_out), arr(params_out) if n_out > 0 else None, n_out)
        self._ref = ctypes.byref(self._st)
        self._group = group
        self._stream = _stream(stream)
        self._fn = _lib.fsdp_sharded_step

    def __call__(self, step: int) -> None:
        self._hp.step = step
        status = self._fn(self._pp, self._ref, self._group, self._stream)
        if status != SS_OK:
            _check("fsdp_sharded_step", status)


def ddp_bucket_pack_average(rank_grads: Sequence[Sequence], bucket_cap_bytes: int,
                            avg_out: Sequence, numels: Optional[Sequence[int]] = None,
                            stream=None) -> int:
    """rank_grads[r][t]: rank r's gradient of tensor t. Returns the bucket count."""
    N = len(rank_grads)
    T = len(avg_out)
    if numels is None:
        numels = [int(t.numel()) for t in avg_out]
    flat = [g for rank in rank_grads for g in rank]
    nb = ctypes.c_int()
    _check("ddp_bucket_pack_average", _lib.ddp_bucket_pack_average(
        N, T, _i64_array(numels), _ptr_array(flat), bucket_cap_bytes, _ptr_array(avg_out),
        ctypes.byref(nb), _stream(stream)))
    return nb.value


def ddp_bucket_pack_average_noalloc(rank_grads: Sequence[Sequence], bucket_cap_bytes: int,
                                    avg_out: Sequence, numels: Optional[Sequence[int]] = None,
                                    stream=None) -> int:
    """Same as ddp_bucket_pack_average, for callers that cannot allocate device
    memory: the library's fixed device array holds the per-call table (at most
    SS_DDP_NOALLOC_TABLE_BYTES; larger requests raise with SS_ESCRATCH).  Calls
    share that array, so calls that could overlap on the GPU must be ordered by
    the caller.  Returns the bucket count."""
    N = len(rank_grads)
    T = len(avg_out)
    if numels is None:
        numels = [int(t.numel()) for t in avg_out]
    flat = [g for rank in rank_grads for g in rank]
    nb = ctypes.c_int()
    _check("ddp_bucket_pack_average_noalloc", _lib.ddp_bucket_pack_average_noalloc(
        N, T, _i64_array(numels), _ptr_array(flat), bucket_cap_bytes, _ptr_array(avg_out),
        ctypes.byref(nb), _stream(stream)))
    return nb.value


def ddp_bucket_assign(numels: Sequence[int], elem_bytes: int, bucket_cap_bytes: int):
    T = len(numels)
    out = (ctypes.c_int * max(1, T))()
    nb = _lib.ddp_bucket_assign(T, _i64_array(numels), elem_bytes, bucket_cap_bytes, out)
    if nb < 0:
        _check("ddp_bucket_assign", nb)
    return [int(out[t]) for t in range(T)], int(nb)
