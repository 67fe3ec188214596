"""GPU parity of the step variants through the C ABI: the AdamW recipe without
fp32 master weights, and gradient accumulation over micro-batches."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_common import Setup
from tests.helpers import check_adamw_state, check_bf16_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    return ss


def _hp(step):
    hp = W.adamw_hparams(step)
    return {k: hp[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay")}


def _packed_grads(ss, su, seed_shift=0):
    ps = su.ps
    ps2 = W.ParamSet(ps.names, ps.shapes, ps.groups, ps.world_size, ps.layout, ps.dtype,
                     seed=ps.seed + 101 * seed_shift, uniform=ps.uniform, grad_std=ps.grad_std)
    out = []
    for rank in W.make_rank_grads(ps2):
        b = torch.empty(su.total, dtype=ps.dtype, device="cuda")
        ss.fsdp_pack(su.plan, [g.cuda() for g in rank], b)
        out.append(b)
    return out


def _oracle_rs(su, bufs):
    return oracle.reduce_scatter(su.N, su.info.shard_numel, [to_np(b) for b in bufs])


NOMASTER = [("tiny_mlp", W.tiny_mlp(2, W.FLAT_ORIG_TRUE)),
            ("awkward1d_false_N7_bf16", W.awkward_1d(7, W.FLAT_ORIG_FALSE, torch.bfloat16)),
            ("awkward1d_true_N5_f32", W.awkward_1d(5, W.FLAT_ORIG_TRUE, torch.float32)),
            ("small_llama_N8", W.llama_1b2(world_size=8, layers=2, hidden=48, ffn=136, vocab=96)),
            ("per_param_N12", W.ParamSet([f"p{i}" for i in range(3)], [(130, 3), (64,), (257, 8)],
                                         [3], 12, W.PER_PARAM_DIM0, torch.bfloat16, seed=11))]


@pytest.mark.parametrize("name,ps", NOMASTER, ids=[c[0] for c in NOMASTER])
def test_no_master_recipe(ss, name, ps):
    su = Setup(ss, ps)
    bf16 = ps.dtype == torch.bfloat16
    shards = torch.empty(su.total, dtype=ps.dtype, device="cuda")
    ss.fsdp_pack(su.plan, su.params, shards)
    m = torch.zeros(su.total, device="cuda")
    v = torch.zeros(su.total, device="cuda")
    grads = _packed_grads(ss, su)
    for step in (1, 2):
        prev_shards, prev_m, prev_v = to_np(shards), to_np(m), to_np(v)
        theta = oracle.bf16_widen(prev_shards) if bf16 else prev_shards.copy()
        ss.fsdp_reduce_scatter_adamw(su.plan, grads, None, m, v, shards,
                                     ss.adamw_params(step=step, **_hp(step)))
        torch.cuda.synchronize()
        g = _oracle_rs(su, grads)
        om, omm, ov = theta.copy(), prev_m.copy(), prev_v.copy()
        o_params = oracle.adamw(g, om, omm, ov, step=step, elem_bytes=2 if bf16 else 4, **_hp(step))
        if bf16:
            # moments as with a master copy; the parameter within one bf16 ulp
            # (plus the master tolerance where the update cancels the weight)
            check_adamw_state(om, to_np(m), to_np(v), om, omm, ov, theta, prev_m, g)
            check_bf16_close(to_np(shards), o_params, om, theta)
        else:
            # fp32 plans: the shard is theta itself
            check_adamw_state(to_np(shards), to_np(m), to_np(v), om, omm, ov, theta, prev_m, g)


@pytest.mark.parametrize("num_micro", [1, 2, 3])
@pytest.mark.parametrize("name,ps", [("small_llama_N8", W.llama_1b2(world_size=8, layers=2, hidden=48,
                                                                    ffn=136, vocab=96)),
                                     ("awkward1d_false_N3", W.awkward_1d(3, W.FLAT_ORIG_FALSE,
                                                                         torch.bfloat16, count=40,
                                                                         max_len=300)),
                                     ("awkward1d_false_N17", W.awkward_1d(17, W.FLAT_ORIG_FALSE,
                                                                          torch.bfloat16, count=40,
                                                                          max_len=300))],
                         ids=["small_llama_N8", "awkward1d_false_N3", "awkward1d_false_N17"])
def test_gradient_accumulation(ss, name, ps, num_micro):
    su = Setup(ss, ps)
    total = su.total
    shards = torch.empty(total, dtype=torch.bfloat16, device="cuda")
    ss.fsdp_pack(su.plan, su.params, shards)
    master = torch.empty(total, device="cuda")
    m = torch.empty_like(master)
    v = torch.empty_like(master)
    ss.fsdp_init_master(su.plan, shards, master, m, v)
    accum = torch.full((total,), float("nan"), device="cuda")
    red = torch.empty(total, device="cuda")
    micro = [_packed_grads(ss, su, j) for j in range(num_micro)]
    o_acc = None
    prev_master, prev_m, prev_v = to_np(master), to_np(m), to_np(v)
    hp = ss.adamw_params(step=1, **_hp(1))
    for j, grads in enumerate(micro):
        last = j == num_micro - 1
        ss.fsdp_reduce_scatter_accumulate(su.plan, grads, accum, j, num_micro, master, m, v, shards,
                                          hp if last else None, red if last else None)
        torch.cuda.synchronize()
        if num_micro > 1:
            o_acc = oracle.accumulate(su.N, su.info.shard_numel, [to_np(b) for b in grads], o_acc
                                      if j > 0 else None)
            if not last:
                np.testing.assert_array_equal(to_np(accum), o_acc)     # bit-exact accumulator
    if num_micro > 1:
        g = oracle.accumulated_grad(o_acc, num_micro)
    else:
        g = _oracle_rs(su, micro[0])
    np.testing.assert_array_equal(to_np(red), g)                      # bit-exact averaged gradient
    om, omm, ov = prev_master.copy(), prev_m.copy(), prev_v.copy()
    oracle.adamw(g, om, omm, ov, step=1, **_hp(1))
    check_adamw_state(to_np(master), to_np(m), to_np(v), om, omm, ov, prev_master, prev_m, g)


def test_accumulation_per_group_and_scalar_tails(ss):
    # groups whose bases are not multiples of 8 elements take the scalar head/tail path
    ps = W.ParamSet([f"p{i}" for i in range(4)], [(5,), (3,), (11,), (2,)], [1, 1, 1, 1], 3,
                    W.FLAT_ORIG_FALSE, torch.bfloat16, seed=5)
    su = Setup(ss, ps)
    micro = [_packed_grads(ss, su, j) for j in range(3)]
    accum = torch.zeros(su.total, device="cuda")
    red = torch.zeros(su.total, device="cuda")
    master = torch.ones(su.total, device="cuda") * 0.01
    m = torch.zeros(su.total, device="cuda")
    v = torch.zeros(su.total, device="cuda")
    shards = torch.zeros(su.total, dtype=torch.bfloat16, device="cuda")
    hp = ss.adamw_params()
    for j, grads in enumerate(micro):
        for g in range(4):
            ss.fsdp_reduce_scatter_accumulate(su.plan, grads, accum, j, 3, master, m, v, shards,
                                              hp if j == 2 else None, red if j == 2 else None,
                                              group=g)
    torch.cuda.synchronize()
    o_acc = None
    for j, grads in enumerate(micro[:2]):
        o_acc = oracle.accumulate(su.N, su.info.shard_numel, [to_np(b) for b in grads], o_acc)
    o_acc = oracle.accumulate(su.N, su.info.shard_numel, [to_np(b) for b in micro[2]], o_acc)
    np.testing.assert_array_equal(to_np(red), oracle.accumulated_grad(o_acc, 3))


def test_accumulation_argument_errors(ss):
    su = Setup(ss, W.tiny_mlp())
    g = [torch.zeros(su.total, dtype=torch.bfloat16, device="cuda")] * 2
    acc = torch.zeros(su.total, device="cuda")
    for step, k in ((3, 3), (-1, 2), (0, 0)):
        with pytest.raises(ss.ShardStateError) as e:
            ss.fsdp_reduce_scatter_accumulate(su.plan, g, acc, step, k)
        assert e.value.status == ss.SS_EINVAL
    with pytest.raises(ss.ShardStateError) as e:   # last micro-batch needs the optimizer
        ss.fsdp_reduce_scatter_accumulate(su.plan, g, acc, 1, 2)
    assert e.value.status == ss.SS_EINVAL
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_reduce_scatter_accumulate(su.plan, g, acc[1:], 0, 2)
    assert e.value.status == ss.SS_EALIGN
