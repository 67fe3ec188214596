"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Layout, pack, all-gather + unpack, the reduce-scatter and the DDP average are
compared bit for bit; AdamW state within the tolerances in tests/helpers.py
(1e-6 relative to the operands' magnitude; bf16 parameters within one ulp).
Small cases span many CTA ranges and ragged tails; the full-size cases run in
the launch configuration the benchmark times and are checked on sampled
elements (elementwise steps) or by whole-array comparison / round trip
(copies).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_common import Setup, guarded, guards_intact, elem_bytes
from tests.helpers import check_adamw_state, check_bf16_params, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    return ss


def _hp_kwargs(step):
    hp = W.adamw_hparams(step)
    return {k: hp[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay")}


def _small_sets():
    sets = [("tiny_mlp_flat_true_N2", W.tiny_mlp(2, W.FLAT_ORIG_TRUE)),
            # world size 1: the reduce-scatter is the identity, the layouts degenerate
            ("tiny_mlp_flat_false_N1", W.tiny_mlp(1, W.FLAT_ORIG_FALSE)),
            ("awkward2d_perparam_N1", W.awkward_2d(1, count=30, max_rows=200))]
    for N in (3, 5, 7):
        for dt in (torch.bfloat16, torch.float32):
            tag = "bf16" if dt == torch.bfloat16 else "f32"
            sets.append((f"awkward1d_false_N{N}_{tag}", W.awkward_1d(N, W.FLAT_ORIG_FALSE, dt)))
            sets.append((f"awkward1d_true_N{N}_{tag}", W.awkward_1d(N, W.FLAT_ORIG_TRUE, dt)))
            sets.append((f"awkward2d_perparam_N{N}_{tag}", W.awkward_2d(N, dtype=dt)))
    # multi-group model with pads (N=3 does not divide the dims)
    small_llama = W.llama_1b2(world_size=3, layers=3, hidden=40, ffn=72, vocab=100)
    sets.append(("small_llama_groups_N3", small_llama))
    sets.append(("small_llama_groups_N8", W.llama_1b2(world_size=8, layers=2, hidden=48,
                                                       ffn=136, vocab=96)))
    # every segment a whole number of 16-byte vectors: the copy kernels' fast path
    sets.append(("small_llama_aligned_N8", W.llama_1b2(world_size=8, layers=2, hidden=64,
                                                        ffn=128, vocab=64)))
    ex = W.ParamSet(["p1", "p2"], [(3,), (5,)], [2], 4, W.FLAT_ORIG_TRUE, torch.bfloat16, seed=9)
    sets.append(("worked_example_3_5", ex))
    big_n = W.ParamSet([f"p{i}" for i in range(5)], [(130, 3), (64,), (0, 4), (1,), (257, 2)], [5],
                       64, W.PER_PARAM_DIM0, torch.bfloat16, seed=10)
    sets.append(("per_param_N64", big_n))
    # N > 8: the general instances read ranks beyond the first 8 in batches of
    # 8 (one further batch at N = 12, two at N = 17), bf16 and fp32
    for N in (12, 17):
        for dt in (torch.bfloat16, torch.float32):
            tag = "bf16" if dt == torch.bfloat16 else "f32"
            sets.append((f"awkward1d_false_N{N}_{tag}", W.awkward_1d(N, W.FLAT_ORIG_FALSE, dt,
                                                                     count=60)))
    return sets


SMALL = _small_sets()


@pytest.mark.parametrize("name,ps", SMALL, ids=[s[0] for s in SMALL])
def test_pack_is_bit_exact(ss, name, ps):
    su = Setup(ss, ps)
    packed, whole = guarded(su.total, ps.dtype)
    ss.fsdp_pack(su.plan, su.params, packed)
    torch.cuda.synchronize()
    assert guards_intact(whole)
    want = su.oracle_pack(su.params_np())
    np.testing.assert_array_equal(to_np(packed).view(np.uint8), want.view(np.uint8))


@pytest.mark.parametrize("name,ps", SMALL, ids=[s[0] for s in SMALL])
def test_all_gather_unpack_is_bit_exact(ss, name, ps):
    su = Setup(ss, ps)
    g = torch.Generator().manual_seed(123)
    if ps.dtype == torch.bfloat16:
        shards_cpu = torch.randint(-32768, 32767, (su.total,), generator=g,
                                   dtype=torch.int16).view(torch.bfloat16)
    else:
        shards_cpu = torch.randn(su.total, generator=g)
    shards = shards_cpu.cuda()
    for n_out in sorted({1, min(ps.world_size, 9)}):
        outs, wholes = [], []
        for j in range(n_out):
            for p in su.params:
                o, w = guarded(p.numel(), ps.dtype)
                outs.append(o)
                wholes.append(w)
        ss.fsdp_all_gather_unpack(su.plan, shards, outs, n_out=n_out)
        torch.cuda.synchronize()
        assert all(guards_intact(w) for w in wholes)
        want = su.oracle_unpack(to_np(shards_cpu), n_out=n_out)
        n = len(su.params)
        for j in range(n_out):
            for i in range(n):
                np.testing.assert_array_equal(to_np(outs[j * n + i]).view(np.uint8),
                                              want[j][i].view(np.uint8))


@pytest.mark.parametrize("name,ps", SMALL, ids=[s[0] for s in SMALL])
def test_reduce_scatter_adamw_three_steps(ss, name, ps):
    su = Setup(ss, ps)
    N, total, dt = su.N, su.total, ps.dtype
    # parameters -> shards (GPU pack, already checked bit-exact) and fp32 state
    shards = torch.empty(total, dtype=dt, device="cuda")
    ss.fsdp_pack(su.plan, su.params, shards)
    master = torch.empty(total, dtype=torch.float32, device="cuda")
    m = torch.empty_like(master)
    v = torch.empty_like(master)
    ss.fsdp_init_master(su.plan, shards, master, m, v)
    torch.cuda.synchronize()
    o_master, o_m, o_v = oracle.init_master(to_np(shards))
    np.testing.assert_array_equal(to_np(master), o_master)
    assert not to_np(m).any() and not to_np(v).any()

    rank_grads_cpu = W.make_rank_grads(ps)
    packed = []
    for r in range(N):
        buf = torch.empty(total, dtype=dt, device="cuda")
        ss.fsdp_pack(su.plan, [g.cuda() for g in rank_grads_cpu[r]], buf)
        packed.append(buf)
    torch.cuda.synchronize()
    for r in range(N):
        want = su.oracle_pack([to_np(g) for g in rank_grads_cpu[r]])
        np.testing.assert_array_equal(to_np(packed[r]).view(np.uint8), want.view(np.uint8))
    packed_np = [to_np(b) for b in packed]

    for step in (1, 2, 3):
        prev_master, prev_m, prev_v = to_np(master), to_np(m), to_np(v)
        reduced, whole_red = guarded(total, torch.float32)
        hp = ss.adamw_params(step=step, **_hp_kwargs(step))
        ss.fsdp_reduce_scatter_adamw(su.plan, packed, master, m, v, shards, hp, reduced)
        torch.cuda.synchronize()
        assert guards_intact(whole_red)
        # oracle on the GPU's previous state (one-step parity)
        om, omm, ov = prev_master.copy(), prev_m.copy(), prev_v.copy()
        c = su.info.shard_numel
        o_params, o_red = oracle.reduce_scatter_adamw(N, c, packed_np, om, omm, ov, step=step,
                                                      **_hp_kwargs(step))
        np.testing.assert_array_equal(to_np(reduced), o_red)          # bit-exact RS
        check_adamw_state(to_np(master), to_np(m), to_np(v), om, omm, ov, prev_master, prev_m,
                          o_red)
        if dt == torch.bfloat16:
            check_bf16_params(to_np(shards), o_params, to_np(master), om, prev_master)
        else:
            np.testing.assert_array_equal(to_np(shards), to_np(master))
    # pads still zero after three steps: unpack + pack reproduces the shards exactly
    outs = [torch.empty_like(p) for p in su.params]
    ss.fsdp_all_gather_unpack(su.plan, shards, outs)
    repacked = torch.empty_like(shards)
    ss.fsdp_pack(su.plan, outs, repacked)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(repacked).view(np.uint8), to_np(shards).view(np.uint8))


def test_per_group_calls_equal_whole_plan_calls(ss):
    ps = W.llama_1b2(world_size=3, layers=4, hidden=40, ffn=72, vocab=100)
    su = Setup(ss, ps)
    N, total = su.N, su.total
    grads = [torch.randn(total, device="cuda").to(torch.bfloat16) for _ in range(N)]
    base_shards = torch.empty(total, dtype=torch.bfloat16, device="cuda")
    ss.fsdp_pack(su.plan, su.params, base_shards)
    results = []
    for mode in ("whole", "groups"):
        shards = base_shards.clone()
        master = torch.empty(total, device="cuda")
        m = torch.empty_like(master)
        v = torch.empty_like(master)
        red = torch.empty_like(master)
        outs = [torch.empty_like(p) for p in su.params]
        repacked = torch.empty_like(shards)
        hp = ss.adamw_params(step=1)
        if mode == "whole":
            ss.fsdp_init_master(su.plan, shards, master, m, v)
            ss.fsdp_reduce_scatter_adamw(su.plan, grads, master, m, v, shards, hp, red)
            ss.fsdp_all_gather_unpack(su.plan, shards, outs)
            ss.fsdp_pack(su.plan, outs, repacked)
        else:
            for g in range(len(su.groups)):
                ss.fsdp_init_master(su.plan, shards, master, m, v, group=g)
                ss.fsdp_reduce_scatter_adamw(su.plan, grads, master, m, v, shards, hp, red, group=g)
                ss.fsdp_all_gather_unpack(su.plan, shards, outs, group=g)
                ss.fsdp_pack(su.plan, outs, repacked, group=g)
        torch.cuda.synchronize()
        results.append([to_np(t) for t in [shards, master, m, v, red, repacked] + outs])
    for a, b in zip(*results):
        np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8))


def test_unaligned_group_ranges_use_scalar_head_and_tail(ss):
    # groups whose base is not a multiple of 8 elements exercise the scalar head/tail path
    ps = W.ParamSet([f"p{i}" for i in range(4)], [(5,), (3,), (11,), (2,)], [1, 1, 1, 1], 3,
                    W.FLAT_ORIG_FALSE, torch.bfloat16, seed=5)
    su = Setup(ss, ps)
    N, total = su.N, su.total
    grads = [torch.randn(total, device="cuda").to(torch.bfloat16) for _ in range(N)]
    red = torch.zeros(total, device="cuda")
    for g in range(4):
        ss.fsdp_reduce_scatter_adamw(su.plan, grads, None, None, None, None, None, red, group=g)
    torch.cuda.synchronize()
    want = oracle.reduce_scatter(N, su.info.shard_numel, [to_np(x) for x in grads])
    # RS is element-wise over the packed index, so per-group RS over all groups == whole RS
    np.testing.assert_array_equal(to_np(red), want)


def test_fp32_shards_equal_master(ss):
    ps = W.awkward_1d(5, W.FLAT_ORIG_TRUE, torch.float32, count=20, max_len=300)
    su = Setup(ss, ps)
    shards = torch.empty(su.total, device="cuda")
    ss.fsdp_pack(su.plan, su.params, shards)
    master = torch.empty_like(shards)
    m = torch.empty_like(shards)
    v = torch.empty_like(shards)
    ss.fsdp_init_master(su.plan, shards, master, m, v)
    grads = [torch.randn(su.total, device="cuda") for _ in range(5)]
    ss.fsdp_reduce_scatter_adamw(su.plan, grads, master, m, v, shards, ss.adamw_params())
    torch.cuda.synchronize()
    assert torch.equal(shards, master)


# ---------------------------------------------------------------------------
# full sizes, launch configuration of the benchmark
# ---------------------------------------------------------------------------

def _sampled_rs_adamw_check(ss, su, grads, shards, master, m, v, step, samples=1 << 20):
    """One RS+AdamW step over the whole plan, checked on a random sample of elements
    (both steps are element-wise over the packed index, so the oracle computes the
    sampled elements from the gathered inputs exactly as it would in place)."""
    N, total = su.N, su.total
    gen = torch.Generator(device="cuda").manual_seed(77)
    k = (min(samples, total) // N) * N
    idx = torch.randint(0, total, (k,), device="cuda", generator=gen)
    in_master = master[idx].cpu().numpy().copy()
    in_m = m[idx].cpu().numpy().copy()
    in_v = v[idx].cpu().numpy().copy()
    in_g = [to_np(gr[idx]) for gr in grads]
    red = torch.empty(total, device="cuda")
    hp = ss.adamw_params(step=step)
    ss.fsdp_reduce_scatter_adamw(su.plan, grads, master, m, v, shards, hp, red)
    torch.cuda.synchronize()
    om, omm, ov = in_master.copy(), in_m.copy(), in_v.copy()
    o_params, o_red = oracle.reduce_scatter_adamw(N, k // N, in_g, om, omm, ov, step=step,
                                                  **_hp_kwargs(step))
    np.testing.assert_array_equal(red[idx].cpu().numpy(), o_red)
    check_adamw_state(master[idx].cpu().numpy(), m[idx].cpu().numpy(), v[idx].cpu().numpy(), om,
                      omm, ov, in_master, in_m, o_red)
    check_bf16_params(to_np(shards[idx]), o_params, master[idx].cpu().numpy(), om, in_master)


def _full_size_setup(ss, ps):
    su = Setup(ss, ps, make_values=False)
    total, N = su.total, su.N
    shards = torch.empty(total, dtype=torch.bfloat16, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(ps.seed)
    shards.copy_((torch.randn(total, device="cuda", generator=gen) * ps.param_std))
    master = torch.empty(total, device="cuda")
    m = torch.empty_like(master)
    v = torch.empty_like(master)
    ss.fsdp_init_master(su.plan, shards, master, m, v)
    grads = W.make_packed_rank_grads(N, total, ps.grad_std, ps.seed, device="cuda")
    return su, shards, master, m, v, grads


def test_llama_block_4096_full_size(ss):
    ps = W.llama_block_4096()
    su, shards, master, m, v, grads = _full_size_setup(ss, ps)
    for step in (1, 2):
        _sampled_rs_adamw_check(ss, su, grads, shards, master, m, v, step)
    # all-gather + unpack, whole arrays against the oracle
    outs = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in ps.shapes]
    ss.fsdp_all_gather_unpack(su.plan, shards, outs)
    torch.cuda.synchronize()
    want = su.oracle_unpack(to_np(shards))[0]
    for o, w in zip(outs, want):
        np.testing.assert_array_equal(to_np(o), w)
    del grads
    torch.cuda.empty_cache()


def test_llama_1b2_full_size(ss):
    ps = W.llama_1b2()
    su, shards, master, m, v, grads = _full_size_setup(ss, ps)
    assert su.total == 1_364_297_728
    _sampled_rs_adamw_check(ss, su, grads, shards, master, m, v, step=1, samples=1 << 21)
    # all-gather + unpack: round trip at full size, oracle on the root group's small
    # norm and on one block group in full
    outs = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in ps.shapes]
    ss.fsdp_all_gather_unpack(su.plan, shards, outs)
    repacked = torch.empty_like(shards)
    ss.fsdp_pack(su.plan, outs, repacked)
    torch.cuda.synchronize()
    assert torch.equal(repacked.view(torch.int16), shards.view(torch.int16))
    g = 5
    grp = su.groups[g]
    base, span = grp["base"], su.N * grp["shard_numel"]
    a, b = grp["first_param"], grp["first_param"] + grp["num_params"]
    want = oracle.all_gather_unpack(su.kind, su.N, 2, su.d0[a:b], su.inner[a:b],
                                    to_np(shards[base:base + span]))[0]
    for i, w in zip(range(a, b), want):
        np.testing.assert_array_equal(to_np(outs[i]), w)
    del grads, outs, repacked
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# DDP
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [8, 12, 17])
@pytest.mark.parametrize("cap", [64 << 10, 1 << 20, 25 << 20, 1 << 30])
def test_ddp_bucket_average_bit_exact(ss, cap, N):
    ds = W.ddp_grads(world_size=N, n_small=70, small=2048, n_large=6, large=65536 + 8, seed=3)
    grads = W.make_ddp_grads(ds, device="cuda")
    outs, wholes = [], []
    for n in ds.numels:
        o, w = guarded(n, torch.bfloat16)
        outs.append(o)
        wholes.append(w)
    nb = ss.ddp_bucket_pack_average(grads, cap, outs)
    torch.cuda.synchronize()
    assert all(guards_intact(w) for w in wholes)
    assert nb == oracle.ddp_buckets(ds.numels, 2, cap)[1]
    want = oracle.ddp_average([[to_np(g) for g in rank] for rank in grads])
    for o, w in zip(outs, want):
        np.testing.assert_array_equal(to_np(o), w)


def test_ddp_full_size_sampled(ss):
    # the full DDP gradient list (1400 x 2048 + 600 x 4,194,304 bf16 per rank, N=8,
    # 45 GB in and out) at the default 25 MiB cap, in the launch shape the benchmark
    # times; 24 tensors (small and large) compared whole against the oracle
    ds = W.ddp_grads()
    grads = W.make_ddp_grads(ds, device="cuda")
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in ds.numels]
    nb = ss.ddp_bucket_pack_average(grads, 25 << 20, outs)
    torch.cuda.synchronize()
    assert nb == oracle.ddp_buckets(ds.numels, 2, 25 << 20)[1]
    rng = np.random.default_rng(0)
    small = [t for t, n in enumerate(ds.numels) if n == 2048]
    large = [t for t, n in enumerate(ds.numels) if n != 2048]
    pick = list(rng.choice(small, 16, replace=False)) + list(rng.choice(large, 8, replace=False))
    pick += [0, len(ds.numels) - 1]
    for t in pick:
        want = oracle.ddp_average([[to_np(grads[r][t])] for r in range(ds.world_size)])[0]
        np.testing.assert_array_equal(to_np(outs[t]), want)
    del grads, outs
    torch.cuda.empty_cache()


def test_ddp_outputs_complete_for_work_after_the_call(ss):
    # buckets go in reverse registration order, so the large tensor registered
    # last is the first bucket and a tiny one the last; the next bucket's
    # kernel starts before the previous one finishes, and work queued on the
    # stream right after the call must still see every output complete
    N = 8
    numels = [3, 5, 7, 4096, 1 << 24]
    g = torch.Generator(device="cuda").manual_seed(5)
    grads = [[(torch.randn(n, generator=g, device="cuda") * 1e-3).to(torch.bfloat16) for n in numels]
             for _ in range(N)]
    for fn in (ss.ddp_bucket_pack_average, ss.ddp_bucket_pack_average_noalloc):
        outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in numels]
        for o in outs:
            o.view(torch.int16).fill_(0x7FBF)
        torch.cuda.synchronize()
        cap = 64 * 1024 if fn is ss.ddp_bucket_pack_average else 1 << 20
        nb = fn(grads, cap, outs)
        assert nb >= 2
        snap = [o.clone() for o in outs]   # queued behind the call, no synchronize
        torch.cuda.synchronize()
        for a, b in zip(snap, outs):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        want = oracle.ddp_average([[to_np(t) for t in rank] for rank in grads])
        for o, w in zip(outs, want):
            np.testing.assert_array_equal(to_np(o), w)


def test_ddp_misaligned_and_odd_sizes(ss):
    # views offset by one element: pointers congruent across ranks, and not
    rng = np.random.default_rng(1)
    N = 5
    numels = [1, 7, 9, 300, 0, 1025]
    bases = [[torch.randn(n + 3, device="cuda").to(torch.bfloat16) for n in numels] for _ in range(N)]
    grads = [[b[(r + t) % 2: (r + t) % 2 + n] for t, (b, n) in enumerate(zip(bases[r], numels))]
             for r in range(N)]
    outs = [torch.empty(n + 1, dtype=torch.bfloat16, device="cuda")[1:] for n in numels]
    ss.ddp_bucket_pack_average(grads, 100, outs, numels=numels)
    torch.cuda.synchronize()
    want = oracle.ddp_average([[to_np(g) for g in rank] for rank in grads])
    for o, w in zip(outs, want):
        np.testing.assert_array_equal(to_np(o), w)


def test_ddp_mixed_buckets_realigned_and_congruent(ss):
    """N = 8, tensors spanning many 4096-element tiles; every third tensor has
    each rank's gradient at its own offset (0..7 elements) from its output, the
    rest are congruent, and the 256 KiB cap puts both kinds in the same and in
    different buckets.  Bit-exact against the oracle."""
    N = 8
    numels = [70_001, 4096, 129, 33_333, 100_000, 8, 65_536, 12_345, 90_000, 1]
    g = torch.Generator(device="cuda").manual_seed(7)
    grads, outs = [], []
    for r in range(N):
        row = []
        for t, n in enumerate(numels):
            sh = (r + 3 * t) % 8 if t % 3 == 0 else 0
            base = (torch.randn(n + 8, generator=g, device="cuda") * 1e-3).to(torch.bfloat16)
            row.append(base[sh:sh + n])
        grads.append(row)
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in numels]
    nb = ss.ddp_bucket_pack_average(grads, 256 * 1024, outs, numels=numels)
    torch.cuda.synchronize()
    assert nb > 1
    want = oracle.ddp_average([[to_np(x) for x in rank] for rank in grads])
    for o, w in zip(outs, want):
        np.testing.assert_array_equal(to_np(o), w)


# ---------------------------------------------------------------------------
# errors come back as status codes, nothing launched
# ---------------------------------------------------------------------------

def test_device_argument_errors(ss):
    ps = W.tiny_mlp()
    su = Setup(ss, ps)
    packed = torch.empty(su.total + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_pack(su.plan, su.params, packed[1:])
    assert e.value.status == ss.SS_EALIGN
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_pack(su.plan, su.params, packed, group=3)
    assert e.value.status == ss.SS_EINVAL
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_all_gather_unpack(su.plan, packed, su.params, n_out=0)
    assert e.value.status == ss.SS_EINVAL
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_reduce_scatter_adamw(su.plan, [packed, packed], None, None, None, None, None, None)
    assert e.value.status == ss.SS_EINVAL
    bad = ss.adamw_params(step=0)
    f = torch.empty(su.total, device="cuda")
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_reduce_scatter_adamw(su.plan, [packed, packed], f, f, f, packed, bad)
    assert e.value.status == ss.SS_EINVAL
    torch.cuda.synchronize()


def test_empty_plan_is_a_no_op(ss):
    plan = ss.fsdp_plan_create(ss.SS_PER_PARAM_DIM0, 4, 2, [0, 0], [3, 5])
    assert plan.info().total_numel == 0
    x = torch.empty(8, dtype=torch.bfloat16, device="cuda")
    f = torch.empty(8, device="cuda")
    ss.fsdp_pack(plan, [x, x], x)
    ss.fsdp_reduce_scatter_adamw(plan, [x] * 4, f, f, f, x, ss.adamw_params())
    ss.fsdp_all_gather_unpack(plan, x, [x, x])
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# pointer-table windows, maximum replica count, the one-group shorthand
# ---------------------------------------------------------------------------

def test_all_gather_windows_and_max_replicas(ss):
    # 200 params x 11 replicas = 2200 pointers > 2048: the call splits into windows
    ps = W.awkward_1d(5, W.FLAT_ORIG_TRUE, torch.bfloat16)
    su = Setup(ss, ps)
    g = torch.Generator().manual_seed(5)
    shards_cpu = torch.randint(-32768, 32767, (su.total,), generator=g,
                               dtype=torch.int16).view(torch.bfloat16)
    shards = shards_cpu.cuda()
    want = su.oracle_unpack(to_np(shards_cpu), n_out=1)[0]
    for n_out in (11, ss.SS_MAX_REPLICAS):
        outs = [torch.empty_like(p) for _ in range(n_out) for p in su.params]
        ss.fsdp_all_gather_unpack(su.plan, shards, outs, n_out=n_out)
        torch.cuda.synchronize()
        n = len(su.params)
        for j in (0, n_out // 2, n_out - 1):
            for i in range(n):
                np.testing.assert_array_equal(to_np(outs[j * n + i]), want[i])
    with pytest.raises(ss.ShardStateError):
        ss.fsdp_all_gather_unpack(su.plan, shards, outs, n_out=ss.SS_MAX_REPLICAS + 1)


def test_pack_more_than_2048_params(ss):
    ps = W.awkward_1d(3, W.FLAT_ORIG_FALSE, torch.bfloat16, count=2300, max_len=40, seed=8)
    su = Setup(ss, ps)
    packed = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
    ss.fsdp_pack(su.plan, su.params, packed)
    outs = [torch.empty_like(p) for p in su.params]
    ss.fsdp_all_gather_unpack(su.plan, packed, outs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(packed), su.oracle_pack(su.params_np()))
    for o, p in zip(outs, su.params_np()):
        np.testing.assert_array_equal(to_np(o), p)


def test_pack_windows_with_pads(ss):
    """More parameters than one pointer table, so pack runs in parameter
    windows, and pads in most rank chunks (PER_PARAM_DIM0, N = 3, dim 0 not a
    multiple of 3): the pad tiles ride with the last window's launch, and
    every one must be zeroed over a buffer of NaN sentinels."""
    shapes = [(1 + (13 * i) % 11, 1 + i % 3) for i in range(2300)]
    ps = W.ParamSet([f"p{i}" for i in range(2300)], shapes, [1000, 1300], 3, W.PER_PARAM_DIM0,
                    torch.bfloat16, seed=9)
    su = Setup(ss, ps)
    assert su.info.pad_numel > 1000
    packed, whole = guarded(su.total, torch.bfloat16)
    ss.fsdp_pack(su.plan, su.params, packed)
    torch.cuda.synchronize()
    assert guards_intact(whole)
    np.testing.assert_array_equal(to_np(packed), su.oracle_pack(su.params_np()))


def test_one_group_shorthand_matches_create(ss):
    ps = W.awkward_2d(5)
    d0, inner = ps.dim0_inner()
    a = ss.fsdp_plan_layout(ss.SS_PER_PARAM_DIM0, 5, 2, d0, inner)
    b = ss.fsdp_plan_create(ss.SS_PER_PARAM_DIM0, 5, 2, d0, inner)
    assert a.info().as_dict() == b.info().as_dict()
    for i in (0, 57, 199):
        assert ss.fsdp_plan_param_offset(a, i) == ss.fsdp_plan_param_offset(b, i)


# ---------------------------------------------------------------------------
# special values: subnormals, infinities, NaN, values near the bf16 / fp32 limits
# ---------------------------------------------------------------------------

def _special_bf16(n, seed):
    """bf16 bit patterns mixing ordinary values with subnormals, +-0, +-inf, NaN and
    values near the largest finite bf16."""
    rng = np.random.default_rng(seed)
    normal = torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).to(torch.bfloat16)
    bits = normal.view(torch.int16).numpy().view(np.uint16).copy()
    specials = np.array([0x0001, 0x8001, 0x007F, 0x807F, 0x0000, 0x8000, 0x7F80, 0xFF80,
                         0x7FC0, 0x7F7F, 0xFF7F, 0x0080, 0x8080], np.uint16)
    pick = rng.random(n) < 0.05
    bits[pick] = rng.choice(specials, int(pick.sum()))
    return bits


def test_special_values_reduce_scatter_and_adamw(ss):
    N, c = 8, 4096 + 5
    total = N * c
    plan = ss.fsdp_plan_layout(ss.SS_FLAT_ORIG_FALSE, N, 2, [total])
    g_np = [_special_bf16(total, 100 + r) for r in range(N)]
    grads = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda() for b in g_np]
    # state: ordinary values plus subnormal / zero masters
    rng = np.random.default_rng(7)
    master_np = rng.normal(0, 0.02, total).astype(np.float32)
    master_np[::97] = np.float32(1e-40)           # subnormal fp32
    master_np[::101] = 0.0
    m_np = np.zeros(total, np.float32)
    v_np = np.zeros(total, np.float32)
    master = torch.from_numpy(master_np.copy()).cuda()
    m = torch.zeros(total, device="cuda")
    v = torch.zeros(total, device="cuda")
    shards = torch.empty(total, dtype=torch.bfloat16, device="cuda")
    red = torch.empty(total, device="cuda")
    hp = ss.adamw_params(step=1)
    ss.fsdp_reduce_scatter_adamw(plan, grads, master, m, v, shards, hp, red)
    torch.cuda.synchronize()
    want = oracle.reduce_scatter(N, c, g_np)
    got = to_np(red)
    nan_w, nan_g = np.isnan(want), np.isnan(got)
    np.testing.assert_array_equal(nan_w, nan_g)                         # NaN exactly where expected
    np.testing.assert_array_equal(got[~nan_w].view(np.uint32),          # everything else bit-exact,
                                  want[~nan_w].view(np.uint32))         # subnormals and infinities included
    om, omm, ov = master_np.copy(), m_np.copy(), v_np.copy()
    o_params = oracle.adamw(want, om, omm, ov, step=1, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                            weight_decay=0.01)
    finite = np.isfinite(want) & np.isfinite(om) & np.isfinite(omm) & np.isfinite(ov)
    gm, gmm, gv = to_np(master), to_np(m), to_np(v)
    # non-finite results appear in the same places on both sides
    np.testing.assert_array_equal(np.isfinite(gm), np.isfinite(om))
    np.testing.assert_array_equal(np.isnan(gmm), np.isnan(omm))
    check_adamw_state(gm[finite], gmm[finite], gv[finite], om[finite], omm[finite], ov[finite],
                      master_np[finite], m_np[finite], want[finite])
    # where the update is finite the bf16 parameter is the rounding of the master
    fin = np.isfinite(gm)
    np.testing.assert_array_equal(to_np(shards)[fin], oracle.bf16_round(gm[fin]))


def _same_or_both_nan(x, y):
    """Bit-identical where either side is a number; NaN in the same places."""
    x, y = np.asarray(x), np.asarray(y)
    if x.dtype == np.uint16:  # bf16 bits
        nx = ((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)
        ny = ((y & 0x7F80) == 0x7F80) & ((y & 0x7F) != 0)
    else:
        nx, ny = np.isnan(x), np.isnan(y)
    np.testing.assert_array_equal(nx, ny)
    np.testing.assert_array_equal(x[~nx].view(np.uint8), y[~ny].view(np.uint8))


@pytest.mark.parametrize("N", [2, 4, 6, 8])
def test_special_values_one_pass_step(ss, N):
    # subnormal rank sums, infinities and NaN through the one pass: its
    # reduced gradient must be the oracle's reduce-scatter, and its state,
    # shards and outputs those of the two calls
    c = 2048 + 3
    total = N * c
    plan = ss.fsdp_plan_layout(ss.SS_FLAT_ORIG_FALSE, N, 2, [total])
    g_np = [_special_bf16(total, 200 + 7 * N + r) for r in range(N)]
    grads = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda() for b in g_np]
    rng = np.random.default_rng(8)
    master_np = rng.normal(0, 0.02, total).astype(np.float32)
    master_np[::97] = np.float32(1e-40)
    runs = []
    for one_pass in (False, True):
        master = torch.from_numpy(master_np.copy()).cuda()
        m = torch.zeros(total, device="cuda")
        v = torch.zeros(total, device="cuda")
        shards = torch.empty(total, dtype=torch.bfloat16, device="cuda")
        red = torch.empty(total, device="cuda")
        out = torch.empty(total, dtype=torch.bfloat16, device="cuda")
        hp = ss.adamw_params(step=1)
        if one_pass:
            ss.fsdp_sharded_step(plan, master, m, v, shards, hp, rank_grads=grads, params_out=[out],
                                 n_out=1, reduced_grad_out=red)
        else:
            ss.fsdp_reduce_scatter_adamw(plan, grads, master, m, v, shards, hp, red)
            ss.fsdp_all_gather_unpack(plan, shards, [out], n_out=1)
        torch.cuda.synchronize()
        runs.append([to_np(t) for t in (red, master, m, v, shards, out)])
    want = oracle.reduce_scatter(N, c, g_np)
    for got in (runs[0][0], runs[1][0]):
        _same_or_both_nan(got, want)
    for x, y in zip(runs[0], runs[1]):
        _same_or_both_nan(x, y)
    assert np.isnan(want).any() and (np.abs(want[np.isfinite(want)]) < 1.2e-38).any()


def test_special_values_ddp_average(ss):
    N, T = 5, 7
    numels = [1, 9, 64, 100, 3, 1031, 8]
    g_np = [[_special_bf16(n, 1000 * r + t) for t, n in enumerate(numels)] for r in range(N)]
    grads = [[torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda() for b in rank]
             for rank in g_np]
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in numels]
    ss.ddp_bucket_pack_average(grads, 128, outs)
    torch.cuda.synchronize()
    want = oracle.ddp_average(g_np)
    for o, w in zip(outs, want):
        got = to_np(o)
        wn = ((w & 0x7F80) == 0x7F80) & ((w & 0x7F) != 0)
        gn = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
        np.testing.assert_array_equal(wn, gn)          # NaN in the same places (payload free)
        np.testing.assert_array_equal(got[~wn], w[~wn])
