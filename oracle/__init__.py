"""CPU oracle for the FSDP / ZeRO-3 sharded-state step.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product package ``sharded_state_gb300`` never imports it, and the two share no
code: the arithmetic here lives in ``ss_oracle.c`` (plain C loops, built with
``-ffp-contract=off``), in ``ledger.py`` (closed forms) and in
``dp_equivalence.py`` (fp64 MLP gradients); this module only marshals numpy
arrays into those C functions.

Element types: bf16 data travels as ``numpy.uint16`` bit patterns, fp32 as
``numpy.float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ss_oracle.c")
_LIB = os.path.join(_HERE, "libssoracle.so")

FLAT_ORIG_FALSE = 0
FLAT_ORIG_TRUE = 1
PER_PARAM_DIM0 = 2

_lib = None


def compile_library(src: str, out: str) -> str:
    """gcc, -O2, no FMA contraction, OpenMP if present: src (C) -> shared library out."""
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_library(_SRC, _LIB)


# SSO_ORACLE_LIB names another build of ss_oracle.c to load instead; the
# mutation tests use it to run the pins against oracles with planted mistakes.
ORACLE_LIB_ENV = "SSO_ORACLE_LIB"


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get(ORACLE_LIB_ENV)
    if not path:
        path = build()
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    vp = ctypes.c_void_p
    lib.sso_layout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i64p, i64p,
                               i64p, i64p, i64p, i64p]
    lib.sso_layout.restype = ctypes.c_int
    lib.sso_pack.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i64p, i64p,
                             ctypes.POINTER(vp), vp]
    lib.sso_pack.restype = ctypes.c_int
    lib.sso_all_gather_unpack.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          i64p, i64p, vp, ctypes.POINTER(vp), ctypes.c_int]
    lib.sso_all_gather_unpack.restype = ctypes.c_int
    lib.sso_reduce_scatter.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                       ctypes.POINTER(vp), vp]
    lib.sso_reduce_scatter.restype = None
    dbl = ctypes.c_double
    lib.sso_adamw.argtypes = [ctypes.c_int64, vp, vp, vp, vp, vp, ctypes.c_int, dbl, dbl, dbl,
                              dbl, dbl, ctypes.c_int64]
    lib.sso_adamw.restype = None
    lib.sso_reduce_scatter_adamw.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                             ctypes.POINTER(vp), vp, vp, vp, vp, vp, dbl, dbl,
                                             dbl, dbl, dbl, ctypes.c_int64]
    lib.sso_reduce_scatter_adamw.restype = None
    lib.sso_accumulate.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(vp),
                                   vp, ctypes.c_int]
    lib.sso_accumulate.restype = None
    lib.sso_accumulated_grad.argtypes = [ctypes.c_int64, vp, ctypes.c_int, vp]
    lib.sso_accumulated_grad.restype = None
    lib.sso_init_master.argtypes = [ctypes.c_int64, vp, ctypes.c_int, vp, vp, vp]
    lib.sso_init_master.restype = None
    lib.sso_ddp_buckets.argtypes = [ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int64,
                                    ctypes.POINTER(ctypes.c_int)]
    lib.sso_ddp_buckets.restype = ctypes.c_int
    lib.sso_ddp_average.argtypes = [ctypes.c_int, ctypes.c_int, i64p, ctypes.POINTER(vp),
                                    ctypes.POINTER(vp)]
    lib.sso_ddp_average.restype = None
    lib.sso_bf16_round.argtypes = [ctypes.c_int64, vp, vp]
    lib.sso_bf16_widen.argtypes = [ctypes.c_int64, vp, vp]
    lib.sso_set_threads.argtypes = [ctypes.c_int]
    lib.sso_get_threads.restype = ctypes.c_int
    lib.sso_has_openmp.restype = ctypes.c_int
    _lib = lib
    return lib


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _ptr(a: np.ndarray):
    return ctypes.cast(a.ctypes.data, ctypes.POINTER(ctypes.c_int64))


def _vp(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _vparr(arrs: Sequence[np.ndarray]):
    arr = (ctypes.c_void_p * max(1, len(arrs)))()
    for k, a in enumerate(arrs):
        arr[k] = a.ctypes.data
    return arr


def _np_dtype(elem_bytes: int):
    return np.uint16 if elem_bytes == 2 else np.float32


def set_threads(n: int) -> None:
    _load().sso_set_threads(int(n))


def get_threads() -> int:
    return int(_load().sso_get_threads())


def has_openmp() -> bool:
    return bool(_load().sso_has_openmp())


# ---------------------------------------------------------------------------
# layout / pack / unpack
# ---------------------------------------------------------------------------

def layout(kind: int, world_size: int, elem_bytes: int, dim0: Sequence[int],
           inner: Optional[Sequence[int]] = None) -> dict:
    """Layout of one group: per-param offsets, chunk rows, shard size."""
    lib = _load()
    n = len(dim0)
    d0 = _i64(dim0 if n else [0])
    inn = _i64(inner) if inner is not None and n else None
    off = np.zeros(max(n, 1), np.int64)
    rows = np.zeros(max(n, 1), np.int64)
    c = np.zeros(1, np.int64)
    L = np.zeros(1, np.int64)
    rc = lib.sso_layout(kind, world_size, elem_bytes, n, _ptr(d0),
                        _ptr(inn) if inn is not None else None, _ptr(off), _ptr(rows), _ptr(c),
                        _ptr(L))
    if rc != 0:
        raise ValueError("oracle layout rejected its arguments")
    return {"offsets": off[:n].tolist(), "chunk_rows": rows[:n].tolist(),
            "shard_numel": int(c[0]), "total_numel": int(c[0]) * world_size,
            "unpadded_numel": int(L[0])}


def pack(kind: int, world_size: int, elem_bytes: int, dim0, inner,
         params: Sequence[np.ndarray]) -> np.ndarray:
    """Per-param arrays (flattened, uint16 or float32) -> rank-major packed buffer."""
    lib = _load()
    lay = layout(kind, world_size, elem_bytes, dim0, inner)
    dt = _np_dtype(elem_bytes)
    ps = [np.ascontiguousarray(p.reshape(-1), dtype=dt) for p in params]
    out = np.empty(max(lay["total_numel"], 1), dtype=dt)
    d0 = _i64(dim0 if len(dim0) else [0])
    inn = _i64(inner) if inner is not None and len(dim0) else None
    rc = lib.sso_pack(kind, world_size, elem_bytes, len(ps), _ptr(d0),
                      _ptr(inn) if inn is not None else None, _vparr(ps), _vp(out))
    if rc != 0:
        raise ValueError("oracle pack rejected its arguments")
    return out[:lay["total_numel"]]


def all_gather_unpack(kind: int, world_size: int, elem_bytes: int, dim0, inner,
                      shards: np.ndarray, n_out: int = 1) -> List[List[np.ndarray]]:
    """Rank-major shards -> n_out replicas of the flattened per-param arrays."""
    lib = _load()
    dt = _np_dtype(elem_bytes)
    n = len(dim0)
    numels = [int(d) * (int(inner[i]) if inner is not None else 1) for i, d in enumerate(dim0)]
    outs = [[np.full(max(s, 1), 0xFFFF if dt == np.uint16 else np.nan, dtype=dt) for s in numels]
            for _ in range(n_out)]
    flat = [a for rep in outs for a in rep]
    sh = np.ascontiguousarray(shards, dtype=dt)
    if sh.size == 0:
        sh = np.zeros(1, dt)
    d0 = _i64(dim0 if n else [0])
    inn = _i64(inner) if inner is not None and n else None
    rc = lib.sso_all_gather_unpack(kind, world_size, elem_bytes, n, _ptr(d0),
                                   _ptr(inn) if inn is not None else None, _vp(sh), _vparr(flat),
                                   n_out)
    if rc != 0:
        raise ValueError("oracle all_gather_unpack rejected its arguments")
    return [[a[:s] for a, s in zip(rep, numels)] for rep in outs]


# ---------------------------------------------------------------------------
# reduce-scatter / AdamW
# ---------------------------------------------------------------------------

def reduce_scatter(world_size: int, shard_numel: int, rank_bufs: Sequence[np.ndarray]) -> np.ndarray:
    """N rank-major buffers of N*c elements -> fp32 mean, all shards side by side."""
    lib = _load()
    assert len(rank_bufs) == world_size
    eb = 2 if rank_bufs[0].dtype == np.uint16 else 4
    bufs = [np.ascontiguousarray(b) for b in rank_bufs]
    out = np.empty(max(world_size * shard_numel, 1), np.float32)
    lib.sso_reduce_scatter(world_size, shard_numel, eb, _vparr(bufs), _vp(out))
    return out[:world_size * shard_numel]


def adamw(grad: np.ndarray, master: np.ndarray, exp_avg: np.ndarray, exp_avg_sq: np.ndarray,
          lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, step: int,
          elem_bytes: int = 2):
    """In-place AdamW on fp32 state; returns the new parameter shard (bf16 bits or fp32)."""
    lib = _load()
    for a in (grad, master, exp_avg, exp_avg_sq):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    out = np.empty(max(grad.size, 1), _np_dtype(elem_bytes))
    lib.sso_adamw(grad.size, _vp(grad), _vp(master), _vp(exp_avg), _vp(exp_avg_sq), _vp(out),
                  elem_bytes, lr, beta1, beta2, eps, weight_decay, step)
    return out[:grad.size]


def accumulate(world_size: int, shard_numel: int, rank_bufs: Sequence[np.ndarray],
               accum: Optional[np.ndarray]) -> np.ndarray:
    """One micro-batch of gradient accumulation: returns acc = RS (accum None)
    or accum + RS, fp32, all ranks' shards side by side."""
    lib = _load()
    eb = 2 if rank_bufs[0].dtype == np.uint16 else 4
    total = world_size * shard_numel
    bufs = [np.ascontiguousarray(b) for b in rank_bufs]
    out = np.empty(max(total, 1), np.float32)
    if accum is not None:
        out[:total] = accum
    lib.sso_accumulate(world_size, shard_numel, eb, _vparr(bufs), _vp(out),
                       1 if accum is None else 0)
    return out[:total]


def accumulated_grad(accum: np.ndarray, num_micro: int) -> np.ndarray:
    lib = _load()
    acc = np.ascontiguousarray(accum, dtype=np.float32)
    out = np.empty(max(acc.size, 1), np.float32)
    lib.sso_accumulated_grad(acc.size, _vp(acc), num_micro, _vp(out))
    return out[:acc.size]


def init_master(param_shards: np.ndarray, out=None):
    """Fresh optimizer state of a shard: (master, exp_avg, exp_avg_sq).
    out: optional three contiguous float32 arrays of the shard's size, written
    in place (and returned) instead of new ones."""
    lib = _load()
    eb = 2 if param_shards.dtype == np.uint16 else 4
    n = param_shards.size
    if out is None:
        master = np.empty(max(n, 1), np.float32)
        m = np.empty(max(n, 1), np.float32)
        v = np.empty(max(n, 1), np.float32)
    else:
        master, m, v = out
        for a in out:
            if a.dtype != np.float32 or a.size != n or not a.flags.c_contiguous:
                raise ValueError("init_master: out must be three contiguous float32 arrays of "
                                 "the shard's size")
    ps = np.ascontiguousarray(param_shards)
    lib.sso_init_master(n, _vp(ps), eb, _vp(master), _vp(m), _vp(v))
    return master[:n], m[:n], v[:n]


def reduce_scatter_adamw(world_size: int, shard_numel: int, rank_grads: Sequence[np.ndarray],
                         master: np.ndarray, exp_avg: np.ndarray, exp_avg_sq: np.ndarray,
                         lr: float, beta1: float, beta2: float, eps: float,
                         weight_decay: float, step: int):
    """Full RS + AdamW on a group; updates state in place, returns (param_shards, reduced)."""
    lib = _load()
    eb = 2 if rank_grads[0].dtype == np.uint16 else 4
    total = world_size * shard_numel
    bufs = [np.ascontiguousarray(b) for b in rank_grads]
    params = np.empty(max(total, 1), _np_dtype(eb))
    reduced = np.empty(max(total, 1), np.float32)
    lib.sso_reduce_scatter_adamw(world_size, shard_numel, eb, _vparr(bufs), _vp(master),
                                 _vp(exp_avg), _vp(exp_avg_sq), _vp(params), _vp(reduced),
                                 lr, beta1, beta2, eps, weight_decay, step)
    return params[:total], reduced[:total]


# ---------------------------------------------------------------------------
# DDP
# ---------------------------------------------------------------------------

def ddp_buckets(numels: Sequence[int], elem_bytes: int, cap_bytes: int):
    lib = _load()
    T = len(numels)
    nm = _i64(numels if T else [0])
    bucket_of = (ctypes.c_int * max(T, 1))()
    count = lib.sso_ddp_buckets(T, _ptr(nm), elem_bytes, cap_bytes, bucket_of)
    return [int(bucket_of[t]) for t in range(T)], int(count)


def ddp_average(rank_grads: Sequence[Sequence[np.ndarray]]) -> List[np.ndarray]:
    """rank_grads[r][t] (uint16 bf16 bits) -> per-tensor bf16 mean."""
    lib = _load()
    N = len(rank_grads)
    T = len(rank_grads[0])
    numels = [int(a.size) for a in rank_grads[0]]
    flat_in = [np.ascontiguousarray(rank_grads[r][t], dtype=np.uint16) for r in range(N)
               for t in range(T)]
    outs = [np.empty(max(s, 1), np.uint16) for s in numels]
    nm = _i64(numels if T else [0])
    lib.sso_ddp_average(N, T, _ptr(nm), _vparr(flat_in), _vparr(outs))
    return [o[:s] for o, s in zip(outs, numels)]


# ---------------------------------------------------------------------------
# bf16 helpers
# ---------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(max(x.size, 1), np.uint16)
    lib.sso_bf16_round(x.size, _vp(x), _vp(out))
    return out[:x.size]


def bf16_widen(x: np.ndarray) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    out = np.empty(max(x.size, 1), np.float32)
    lib.sso_bf16_widen(x.size, _vp(x), _vp(out))
    return out[:x.size]
