"""Seeded random plans through every path of the step.

Each case draws the following:
  - a world size and a layout;
  - parameter shapes: empties, single elements, odd and vector-sized lengths, and 1-D or 2-D;
  - a split of the parameters into groups, empty groups included;
  - a 2-byte offset for every per-parameter tensor.

On each case:
  - pack from tensors at their offsets equals the oracle's pack, pads zero;
  - the all-gather into outputs at their own offsets (n_out = 2) equals the parameters;
  - the one-pass step from packed gradients and from the per-parameter gradient sets at their
    offsets (fused copy-in), both over the whole plan and group by group, equals RS + AdamW
    followed by the all-gather bit for bit over two steps;
  - no call writes a byte outside its outputs.

These cases reach plan shapes the fixed cases do not: segments of a few elements, group ranges
inside one 8-element vector, ranks with empty shards, and N > 8 next to misaligned runs.
"""
import random

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_common import SENTINEL_BF16, Setup
from tests.helpers import to_np

pytestmark = pytest.mark.gpu

CASES = 64


@pytest.fixture(scope="module")
def ss():
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    return ss


def _draw(seed):
    rng = random.Random(1000 + seed)
    N = rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 12])
    layout = rng.choice([W.FLAT_ORIG_FALSE, W.FLAT_ORIG_TRUE, W.PER_PARAM_DIM0])
    n = rng.randint(1, 24)
    shapes = []
    for _ in range(n):
        u = rng.random()
        d0 = (0 if u < 0.1 else rng.randint(1, 9) if u < 0.3 else rng.randint(10, 3000)
              if u < 0.85 else rng.randint(3000, 40000))
        if rng.random() < 0.4:
            shapes.append((d0, rng.choice([1, 2, 3, 5, 8, 16])))
        else:
            shapes.append((d0,))
    if all(d[0] == 0 for d in shapes):
        shapes[0] = (rng.randint(1, 100),)
    groups, left = [], n
    while left:
        g = 0 if rng.random() < 0.08 else rng.randint(1, left)
        groups.append(g)
        left -= g
    if rng.random() < 0.2:
        groups.append(0)
    ps = W.ParamSet([f"f{i}" for i in range(n)], shapes, groups, N, layout, torch.bfloat16,
                    seed=seed)
    return ps, rng


def _shifted(numel, shift):
    whole = torch.empty(numel + 16, dtype=torch.bfloat16, device="cuda")
    whole.view(torch.int16).fill_(SENTINEL_BF16)
    return whole[shift:shift + numel], whole


def _intact(view, whole):
    w = to_np(whole)
    s = (view.data_ptr() - whole.data_ptr()) // 2
    return bool((w[:s] == SENTINEL_BF16).all() and (w[s + view.numel():] == SENTINEL_BF16).all())


def _state(ss, su):
    shards = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
    ss.fsdp_pack(su.plan, su.params, shards)
    master = torch.empty(su.total, device="cuda")
    m, v = torch.empty_like(master), torch.empty_like(master)
    ss.fsdp_init_master(su.plan, shards, master, m, v)
    return [shards, master, m, v]


def _hp(ss, step):
    return ss.adamw_params(step=step, **{k: v for k, v in W.adamw_hparams(step).items()
                                         if k != "step"})


@pytest.mark.parametrize("seed", range(CASES))
def test_random_plan(ss, seed):
    ps, rng = _draw(seed)
    su = Setup(ss, ps)
    N, n, G = su.N, len(su.params), len(ps.groups)
    numels = [p.numel() for p in su.params]
    wholes = []

    def views(tensors=None, count=None):
        out = []
        for i in range(count if count is not None else len(tensors)):
            k = numels[i % n]
            v, w = _shifted(k, rng.randint(0, 7))
            if tensors is not None:
                v.copy_(tensors[i].reshape(-1))
            out.append(v)
            wholes.append((v, w))
        return out

    # pack from offset tensors
    packed = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
    ss.fsdp_pack(su.plan, views([p for p in su.params]), packed)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(packed), su.oracle_pack(su.params_np()))
    # all-gather into offset outputs, two replicas
    outs = views(count=2 * n)
    ss.fsdp_all_gather_unpack(su.plan, packed, outs, n_out=2)
    torch.cuda.synchronize()
    for j in range(2):
        for i, p in enumerate(su.params_cpu):
            np.testing.assert_array_equal(to_np(outs[j * n + i]), to_np(p))
    # the step along every path
    grads_cpu = W.make_rank_grads(ps)
    gpk = []
    for r in range(N):
        b = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, [g.cuda() for g in grads_cpu[r]], b)
        gpk.append(b)
    gpp = views([g for rank in grads_cpu for g in rank])
    modes = ["two_calls", "packed", "copy_in", "packed_groups", "copy_in_groups"]
    state = {m: _state(ss, su) for m in modes}
    o = {m: (views(count=n) if m != "two_calls" else
             [torch.empty(k, dtype=torch.bfloat16, device="cuda") for k in numels]) for m in modes}
    for step in (1, 2):
        hp = _hp(ss, step)
        for m in modes:
            sh, ma, mm, vv = state[m]
            src = {"rank_grads": gpk} if m.startswith("packed") else {"rank_param_grads": gpp}
            if m == "two_calls":
                ss.fsdp_reduce_scatter_adamw(su.plan, gpk, ma, mm, vv, sh, hp)
                ss.fsdp_all_gather_unpack(su.plan, sh, o[m], n_out=1)
            elif m.endswith("groups"):
                for g in range(G):
                    ss.fsdp_sharded_step(su.plan, ma, mm, vv, sh, hp, params_out=o[m], n_out=1,
                                         group=g, **src)
            else:
                ss.fsdp_sharded_step(su.plan, ma, mm, vv, sh, hp, params_out=o[m], n_out=1, **src)
        torch.cuda.synchronize()
        want = [to_np(t).view(np.uint8) for t in state["two_calls"]]
        want_o = [to_np(t) for t in o["two_calls"]]
        for m in modes[1:]:
            for x, y in zip(state[m], want):
                np.testing.assert_array_equal(to_np(x).view(np.uint8), y, err_msg=m)
            for x, y in zip(o[m], want_o):
                np.testing.assert_array_equal(to_np(x), y, err_msg=m)
    for v, w in wholes:
        assert _intact(v, w)


@pytest.mark.parametrize("seed", range(16))
def test_random_plan_parameter_windows(ss, seed):
    # more parameters x pointers than one kernel-parameter table holds (2048):
    # the one pass runs window by window over the packed runs of each window's
    # segments, and must still equal the two calls bit for bit
    rng = random.Random(5000 + seed)
    N = rng.choice([2, 3, 7, 8, 12])
    layout = rng.choice([W.FLAT_ORIG_FALSE, W.FLAT_ORIG_TRUE, W.PER_PARAM_DIM0])
    n = rng.randint(90, 160)
    shapes = [(rng.choice([0, 1, 3, 8, 17, rng.randint(1, 3000)]),) for _ in range(n)]
    shapes[0] = (rng.randint(100, 3000),)
    cuts = sorted(rng.sample(range(1, n), rng.randint(0, 6)))
    groups = [b - a for a, b in zip([0] + cuts, cuts + [n])]
    ps = W.ParamSet([f"w{i}" for i in range(n)], shapes, groups, N, layout, torch.bfloat16,
                    seed=seed + 77)
    su = Setup(ss, ps)
    n_out = 24  # 24 (packed) or N + 24 (copy-in) pointers per parameter: windows of <= 85
    numels = [p.numel() for p in su.params]
    grads_cpu = W.make_rank_grads(ps)
    gpk = []
    for r in range(N):
        b = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, [g.cuda() for g in grads_cpu[r]], b)
        gpk.append(b)
    gpp = [g.cuda().reshape(-1) for rank in grads_cpu for g in rank]
    hp = _hp(ss, 1)
    sa = _state(ss, su)
    outs_a = [torch.empty(k, dtype=torch.bfloat16, device="cuda") for _ in range(n_out) for k in numels]
    ss.fsdp_reduce_scatter_adamw(su.plan, gpk, sa[1], sa[2], sa[3], sa[0], hp)
    ss.fsdp_all_gather_unpack(su.plan, sa[0], outs_a, n_out=n_out)
    for src in ({"rank_grads": gpk}, {"rank_param_grads": gpp}):
        sb = _state(ss, su)
        outs_b = [torch.empty(k, dtype=torch.bfloat16, device="cuda") for _ in range(n_out)
                  for k in numels]
        ss.fsdp_sharded_step(su.plan, sb[1], sb[2], sb[3], sb[0], hp, params_out=outs_b,
                             n_out=n_out, **src)
        torch.cuda.synchronize()
        for x, y in zip(sa, sb):
            np.testing.assert_array_equal(to_np(x).view(np.uint8), to_np(y).view(np.uint8))
        for x, y in zip(outs_a, outs_b):
            np.testing.assert_array_equal(to_np(x), to_np(y))
