"""The allocation-free DDP entry point, checked against the allocating one.

Some callers cannot allocate device memory at all -- a framework that owns
every byte through its own allocator, a latency-critical loop that must not
grow a memory pool, a process at its memory limit -- so the library offers
ddp_bucket_pack_average_noalloc, whose per-call table lives in a fixed device
array inside the library.  This file is collected last on purpose: it runs
after every other test (sharing the process and the array with them) and also
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    return ss


def _bits(t):
    return t.reshape(-1).cpu().view(torch.int16).numpy()


def _call_noalloc(ss, grads, cap, outs):
    """Straight through the C ABI (no binding helper)."""
    N, T = len(grads), len(outs)
    numels = (ctypes.c_int64 * T)(*[o.numel() for o in outs])
    flat = (ctypes.c_void_p * (N * T))(*[g.data_ptr() for rank in grads for g in rank])
    outp = (ctypes.c_void_p * T)(*[o.data_ptr() for o in outs])
    nb = ctypes.c_int()
    st = ss.lib().ddp_bucket_pack_average_noalloc(
        N, T, numels, flat, cap, outp, ctypes.byref(nb),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, nb.value


def test_noalloc_matches_allocating_entry_point_two_calls(ss):
    for call, seed in enumerate((3, 4)):
        ds = W.ddp_grads(world_size=8, n_small=90, small=2048, n_large=5, large=40000 + 8 * call,
                         seed=seed)
        grads = W.make_ddp_grads(ds, device="cuda")
        cap = 256 << 10
        want = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in ds.numels]
        got = [torch.full((n,), float("nan"), dtype=torch.bfloat16, device="cuda")
               for n in ds.numels]
        nb_want = ss.ddp_bucket_pack_average(grads, cap, want)
        st, nb_got = _call_noalloc(ss, grads, cap, got)
        torch.cuda.synchronize()
        assert st == ss.SS_OK, ss.ss_strerror(st)
        assert nb_got == nb_want > 1
        for a, b in zip(got, want):
            # the DDP average is bit-exact between the two entry points
            np.testing.assert_array_equal(_bits(a), _bits(b))


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
