"""Host-side tests of libshardstate (no GPU needed): the library loads, exports
every symbol the header declares, its planner agrees with the oracle's
(independently written) planner, and argument errors come back as status
codes before anything is launched."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import header_functions


@pytest.fixture(scope="module")
def ss():
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    return ss


def test_library_exports_every_header_symbol(ss):
    names = header_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(ss.lib(), name), name
    assert set(names) == set(ss.EXPORTED)
    assert ss.ss_version() == "0.1.0"
    assert ss.ss_strerror(ss.SS_EALIGN) == "pointer misaligned"


def _compare_plan(ss, kind, N, eb, dim0, inner=None, groups=None):
    plan = ss.fsdp_plan_create(kind, N, eb, dim0, inner, group_num_params=groups, host_only=True)
    info = plan.info()
    assert info.has_device_metadata == 0
    gsizes = groups or [len(dim0)]
    lo = 0
    base = 0
    total_unpadded = 0
    for g, cnt in enumerate(gsizes):
        lay = oracle.layout(kind, N, eb, dim0[lo:lo + cnt],
                            inner[lo:lo + cnt] if inner is not None else None)
        grp = ss.fsdp_plan_group(plan, g)
        assert grp["base"] == base and grp["shard_numel"] == lay["shard_numel"]
        assert grp["first_param"] == lo and grp["num_params"] == cnt
        for i in range(cnt):
            off, rows = ss.fsdp_plan_param_offset(plan, lo + i)
            assert off == base + lay["offsets"][i]
            assert rows == lay["chunk_rows"][i]
        base += lay["total_numel"]
        total_unpadded += lay["unpadded_numel"]
        lo += cnt
    assert info.total_numel == base
    assert info.shard_numel * N == base
    assert info.unpadded_numel == total_unpadded
    assert info.pad_numel == base - total_unpadded
    plan.destroy()


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_plan_tables_validate(ss, kind):
    cases = []
    for N in (1, 3, 7, 8, 64):
        if kind == 2:
            ps = W.awkward_2d(N)
            cases.append((N, *ps.dim0_inner(), [1, 0, 37, 62, 100]))
        else:
            ps = W.awkward_1d(N, kind, torch.bfloat16)
            cases.append((N, ps.numels(), None, [1, 0, 37, 62, 100]))
    big = W.llama_1b2()
    if kind == 2:
        cases.append((8, *big.dim0_inner(), big.groups))
    for N, d0, inner, groups in cases:
        for eb in (2, 4):
            for g in (None, groups):
                plan = ss.fsdp_plan_create(kind, N, eb, d0, inner, group_num_params=g,
                                           host_only=True)
                ss.fsdp_plan_validate(plan)
                plan.destroy()


def test_random_plans_validate(ss):
    # the random plans the GPU fuzz cases run (every layout, N up to 12,
    # empty parameters and groups): every table the kernels index through
    # passes the library's own checks, in bf16 and fp32
    from tests.test_gpu_fuzz import _draw
    for seed in range(64):
        ps, _ = _draw(seed)
        d0, inner = ps.dim0_inner()
        for eb in (2, 4):
            plan = ss.fsdp_plan_create(ps.layout, ps.world_size, eb, d0, inner,
                                       group_num_params=ps.groups, host_only=True)
            ss.fsdp_plan_validate(plan)
            plan.destroy()


def test_worked_example_through_the_library(ss):
    for kind, per_rank in ((ss.SS_FLAT_ORIG_FALSE, 2), (ss.SS_FLAT_ORIG_TRUE, 4),
                           (ss.SS_PER_PARAM_DIM0, 3)):
        plan = ss.fsdp_plan_create(kind, 4, 2, [3, 5], host_only=True)
        assert plan.info().shard_numel == per_rank


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("N", [1, 3, 5, 7, 8, 64])
@pytest.mark.parametrize("eb", [2, 4])
def test_planner_matches_oracle_awkward(ss, kind, N, eb):
    dtype = torch.bfloat16 if eb == 2 else torch.float32
    if kind == 2:
        ps = W.awkward_2d(max(N, 1), dtype=dtype)
        d0, inner = ps.dim0_inner()
    else:
        ps = W.awkward_1d(N, kind, dtype)
        d0, inner = ps.numels(), None
    _compare_plan(ss, kind, N, eb, d0, inner)
    # the same params split into uneven groups
    groups = [1, 0, 37, 62, 100]
    _compare_plan(ss, kind, N, eb, d0, inner, groups)


def test_planner_matches_oracle_llama(ss):
    ps = W.llama_1b2()
    d0, inner = ps.dim0_inner()
    _compare_plan(ss, ss.SS_PER_PARAM_DIM0, 8, 2, d0, inner, ps.groups)
    plan = ss.fsdp_plan_create(ss.SS_PER_PARAM_DIM0, 8, 2, d0, inner, ps.groups, host_only=True)
    info = plan.info()
    assert info.unpadded_numel == info.total_numel == 1_364_297_728
    assert info.num_groups == 25
    ps2 = W.llama_block_4096()
    d0, inner = ps2.dim0_inner()
    plan2 = ss.fsdp_plan_create(ss.SS_PER_PARAM_DIM0, 8, 2, d0, inner, host_only=True)
    assert plan2.info().total_numel == 202_383_360


def test_plan_argument_errors(ss):
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_plan_create(5, 4, 2, [3], host_only=True)
    assert e.value.status == ss.SS_EINVAL
    for N in (0, 65):
        with pytest.raises(ss.ShardStateError):
            ss.fsdp_plan_create(0, N, 2, [3], host_only=True)
    with pytest.raises(ss.ShardStateError):
        ss.fsdp_plan_create(0, 4, 3, [3], host_only=True)
    with pytest.raises(ss.ShardStateError):
        ss.fsdp_plan_create(0, 4, 2, [-1], host_only=True)
    with pytest.raises(ss.ShardStateError):  # group sizes must sum to num_params
        ss.fsdp_plan_create(0, 4, 2, [3, 4], group_num_params=[1], host_only=True)
    with pytest.raises(ss.ShardStateError) as e:  # numel beyond int64 / the element cap
        ss.fsdp_plan_create(2, 4, 2, [1 << 40], [1 << 40], host_only=True)
    assert e.value.status == ss.SS_EOVERFLOW
    # empty plan is valid
    plan = ss.fsdp_plan_create(1, 4, 2, [], host_only=True)
    assert plan.info().total_numel == 0


def test_launching_calls_on_host_only_plan_fail_before_launch(ss):
    plan = ss.fsdp_plan_create(1, 2, 2, [16, 16], host_only=True)
    fake = 1 << 20  # never dereferenced: the call must return before touching the device
    arr = (ctypes.c_void_p * 2)(fake, fake)
    st = ss.lib().fsdp_pack(plan, arr, ctypes.c_void_p(fake), -1, None)
    assert st == ss.SS_ENODEVICE
    st = ss.lib().fsdp_all_gather_unpack(plan, ctypes.c_void_p(fake), arr, 1, -1, None)
    assert st == ss.SS_ENODEVICE
    hp = ss.adamw_params()
    st = ss.lib().fsdp_reduce_scatter_adamw(plan, arr, fake, fake, fake, fake, ctypes.byref(hp),
                                            None, -1, None)
    assert st == ss.SS_ENODEVICE
    st = ss.lib().fsdp_init_master(plan, fake, fake, fake, fake, -1, None)
    assert st == ss.SS_ENODEVICE


def test_ddp_bucket_assignment_matches_oracle(ss):
    rng = np.random.default_rng(4)
    for trial in range(200):
        T = int(rng.integers(0, 30))
        numels = [int(x) for x in rng.integers(0, 100, T)]
        cap = int(rng.integers(1, 400))
        got = ss.ddp_bucket_assign(numels, 2, cap)
        want = oracle.ddp_buckets(numels, 2, cap)
        assert got == want
    ds = W.ddp_grads()
    for cap in W.DDP_BUCKET_CAPS:
        assert ss.ddp_bucket_assign(ds.numels, 2, cap) == oracle.ddp_buckets(ds.numels, 2, cap)


def test_ddp_argument_errors_before_launch(ss):
    lib = ss.lib()
    numels = (ctypes.c_int64 * 2)(4, 4)
    ptrs = (ctypes.c_void_p * 4)(1 << 20, 1 << 20, 1 << 20, 1 << 20)
    outs = (ctypes.c_void_p * 2)(1 << 20, 1 << 20)
    nb = ctypes.c_int()
    assert lib.ddp_bucket_pack_average(0, 2, numels, ptrs, 64, outs, ctypes.byref(nb), None) == ss.SS_EINVAL
    assert lib.ddp_bucket_pack_average(2, 2, numels, ptrs, 0, outs, ctypes.byref(nb), None) == ss.SS_EINVAL
    bad = (ctypes.c_void_p * 4)((1 << 20) + 1, 1 << 20, 1 << 20, 1 << 20)
    assert lib.ddp_bucket_pack_average(2, 2, numels, bad, 64, outs, ctypes.byref(nb), None) == ss.SS_EALIGN
    nul = (ctypes.c_void_p * 4)(None, 1 << 20, 1 << 20, 1 << 20)
    assert lib.ddp_bucket_pack_average(2, 2, numels, nul, 64, outs, ctypes.byref(nb), None) == ss.SS_EINVAL
