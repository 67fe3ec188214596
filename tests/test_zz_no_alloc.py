"""The allocation-free DDP entry point, checked against the allocating one and
against the oracle.

Some callers cannot allocate device memory at all -- a framework that owns
every byte through its own allocator, a latency-critical loop that must not
grow a memory pool, a process at its memory limit -- so the library offers
ddp_bucket_pack_average_noalloc, whose per-call table lives in a fixed device
array inside the library.  This file is collected last on purpose: it runs
after every other test, sharing the process and the array with them, and one
test below runs the file again alone in a fresh process.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def ss():
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    return ss


def _bits(t):
    return t.reshape(-1).cpu().view(torch.int16).numpy().view(np.uint16)


def _call(ss, name, grads, cap, outs, stream=None):
    """Straight through the C ABI (no binding helper); returns (status, buckets)."""
    N, T = len(grads), len(outs)
    numels = (ctypes.c_int64 * T)(*[o.numel() for o in outs])
    flat = (ctypes.c_void_p * (N * T))(*[g.data_ptr() for rank in grads for g in rank])
    outp = (ctypes.c_void_p * T)(*[o.data_ptr() for o in outs])
    nb = ctypes.c_int()
    s = stream if stream is not None else torch.cuda.current_stream()
    st = getattr(ss.lib(), name)(N, T, numels, flat, cap, outp, ctypes.byref(nb),
                                 ctypes.c_void_p(s.cuda_stream))
    return st, nb.value


def _call_noalloc(ss, grads, cap, outs, stream=None):
    return _call(ss, "ddp_bucket_pack_average_noalloc", grads, cap, outs, stream)


def _nan_outputs(numels):
    return [torch.full((n,), float("nan"), dtype=torch.bfloat16, device="cuda") for n in numels]


def test_noalloc_matches_allocating_entry_point_two_calls(ss):
    for call, seed in enumerate((3, 4)):
        ds = W.ddp_grads(world_size=8, n_small=90, small=2048, n_large=5, large=40000 + 8 * call,
                         seed=seed)
        grads = W.make_ddp_grads(ds, device="cuda")
        cap = 256 << 10
        want = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in ds.numels]
        got = _nan_outputs(ds.numels)
        nb_want = ss.ddp_bucket_pack_average(grads, cap, want)
        st, nb_got = _call_noalloc(ss, grads, cap, got)
        torch.cuda.synchronize()
        assert st == ss.SS_OK, ss.ss_strerror(st)
        assert nb_got == nb_want > 1
        for a, b in zip(got, want):
            # the DDP average is bit-exact between the two entry points
            np.testing.assert_array_equal(_bits(a), _bits(b))


def test_noalloc_back_to_back_calls_on_one_stream_match_the_oracle(ss):
    """Two calls with different tensor lists queued on one stream with no
    synchronisation between them: the second call rewrites the shared table
    while the first call's buckets may still be running, and the stream's
    order must keep the first call's kernels on its own table.  The first
    list's leading bucket holds a 16M-element tensor, so its kernels are still
    running when the second call is issued; both results are checked against
    the oracle after one synchronisation."""
    lists = [W.ddp_grads(world_size=8, n_small=40, small=2048, n_large=1, large=1 << 24, seed=5),
             W.ddp_grads(world_size=8, n_small=120, small=2048 + 8, n_large=6, large=65536 + 40,
                         seed=6)]
    cap = 1 << 20
    grads = [W.make_ddp_grads(ds, device="cuda") for ds in lists]
    outs = [_nan_outputs(ds.numels) for ds in lists]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        statuses = [_call_noalloc(ss, g, cap, o, stream=s) for g, o in zip(grads, outs)]
    s.synchronize()
    for (st, nb), ds, g, o in zip(statuses, lists, grads, outs):
        assert st == ss.SS_OK, ss.ss_strerror(st)
        assert nb == oracle.ddp_buckets(ds.numels, 2, cap)[1]
        want = oracle.ddp_average([[_bits(t) for t in rank] for rank in g])
        for a, b in zip(o, want):
            np.testing.assert_array_equal(_bits(a), b)


class _PoolProbe:
    """The device's default memory pool (where cudaMallocAsync allocates) and
    the device's free memory, read through the CUDA driver API."""
    USED_MEM_CURRENT, USED_MEM_HIGH = 7, 8  # CUmemPool_attribute

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def _get(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_high(self):
        # setting the high-water mark resets it to the pool's current use
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(zero)) == 0

    def used_high(self):
        return self._get(self.USED_MEM_HIGH)

    def used_now(self):
        return self._get(self.USED_MEM_CURRENT)

    def free_bytes(self):
        free, total = ctypes.c_size_t(), ctypes.c_size_t()
        assert self.cu.cuMemGetInfo_v2(ctypes.byref(free), ctypes.byref(total)) == 0
        return free.value


def test_noalloc_allocates_nothing(ss):
    """The pool's high-water mark stays at its current use across a no-alloc
    call, and the device's free memory is unchanged; the allocating entry
    point, run the same way, does raise the mark (the probe sees
    allocations)."""
    ds = W.ddp_grads(world_size=8, n_small=90, small=2048, n_large=5, large=40000, seed=7)
    grads = W.make_ddp_grads(ds, device="cuda")
    outs = _nan_outputs(ds.numels)
    cap = 256 << 10
    st, _ = _call_noalloc(ss, grads, cap, outs)  # the array's module is loaded by now
    assert st == ss.SS_OK
    torch.cuda.synchronize()
    probe = _PoolProbe()
    base = probe.used_now()
    probe.reset_high()
    free0 = probe.free_bytes()
    for _ in range(3):
        st, _ = _call_noalloc(ss, grads, cap, outs)
        assert st == ss.SS_OK
    torch.cuda.synchronize()
    # (a reset mark reads zero until the next allocation, so <= rather than ==)
    assert probe.used_high() <= base
    assert probe.free_bytes() == free0
    # control: the allocating entry point takes its table from the same pool
    probe.reset_high()
    st, _ = _call(ss, "ddp_bucket_pack_average", grads, cap, outs)
    assert st == ss.SS_OK
    torch.cuda.synchronize()
    assert probe.used_high() > base


# Both calls are refused before they enqueue anything, so the graph is empty.
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_a_capturing_stream_is_refused(ss):
    """Both DDP entry points copy their table from call-local host memory, so
    a stream being captured into a graph gets SS_EINVAL and nothing is
    queued (the captured graph stays empty)."""
    ds = W.ddp_grads(world_size=4, n_small=8, small=2048, n_large=1, large=4096, seed=8)
    grads = W.make_ddp_grads(ds, device="cuda")
    outs = _nan_outputs(ds.numels)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st_noalloc, _ = _call_noalloc(ss, grads, 1 << 20, outs, stream=s)
        st_alloc, _ = _call(ss, "ddp_bucket_pack_average", grads, 1 << 20, outs, stream=s)
    torch.cuda.synchronize()
    assert st_noalloc == ss.SS_EINVAL
    assert st_alloc == ss.SS_EINVAL
    # untouched outputs, and the stream works as before once capture has ended
    assert all(torch.isnan(o.float()).all() for o in outs)
    st, _ = _call_noalloc(ss, grads, 1 << 20, outs)
    torch.cuda.synchronize()
    assert st == ss.SS_OK
    want = oracle.ddp_average([[_bits(t) for t in rank] for rank in grads])
    for a, b in zip(outs, want):
        np.testing.assert_array_equal(_bits(a), b)


def test_noalloc_rejects_tables_beyond_its_array(ss):
    N = 8
    per_tensor = 8 * (N + 1) + 8
    T = ss.SS_DDP_NOALLOC_TABLE_BYTES // per_tensor + 1
    x = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    grads = [[x] * T for _ in range(N)]
    outs = [x] * T
    st, _ = _call_noalloc(ss, grads, 1 << 20, outs)
    assert st == ss.SS_ESCRATCH
    assert ss.ss_strerror(st) == "request exceeds the fixed scratch array"


def test_this_file_alone_in_a_fresh_process():
    """The same tests in a new process whose first use of the array is here."""
    if os.environ.get("SS_NOALLOC_CHILD"):
        pytest.skip("already the fresh process")
    env = dict(os.environ, SS_NOALLOC_CHILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.abspath(__file__), "-x", "-q",
                        "-m", "gpu", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
