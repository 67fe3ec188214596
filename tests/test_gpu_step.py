"""GPU parity of the one-pass step (fsdp_sharded_step) through the C ABI.

The fused kernel runs the same fp32 operations in the same order as
fsdp_reduce_scatter_adamw, so its state and shards must be bit-identical to
the two-call path, and its per-parameter outputs bit-identical to
fsdp_all_gather_unpack of its own shards; both are also checked against the
oracle.  Gradients come either from packed rank buffers or straight from the
per-parameter gradient tensors (fused copy-in) -- the two must agree bit for
bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_common import SENTINEL_BF16, Setup, guarded, guards_intact
from tests.helpers import check_adamw_state, check_bf16_params, to_np

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


CASES = [("tiny_mlp", W.tiny_mlp(2, W.FLAT_ORIG_TRUE)),
         ("awkward1d_false_N7", W.awkward_1d(7, W.FLAT_ORIG_FALSE, torch.bfloat16)),
         ("awkward1d_true_N5", W.awkward_1d(5, W.FLAT_ORIG_TRUE, torch.bfloat16)),
         ("awkward2d_N3", W.awkward_2d(3)),
         # misaligned at N = 1 (one rank: every vector from the single buffer)
         # and N = 16 (ranks beyond the first 8 read one by one)
         ("awkward1d_false_N1", W.awkward_1d(1, W.FLAT_ORIG_FALSE, torch.bfloat16, count=60)),
         ("awkward2d_N16", W.awkward_2d(16, count=60)),
         # misaligned at N = 17 and 24: ranks beyond the first 16 as well
         ("awkward1d_false_N17", W.awkward_1d(17, W.FLAT_ORIG_FALSE, torch.bfloat16, count=60)),
         ("awkward1d_true_N24", W.awkward_1d(24, W.FLAT_ORIG_TRUE, torch.bfloat16, count=60)),
         ("small_llama_N3", W.llama_1b2(world_size=3, layers=3, hidden=40, ffn=72, vocab=100)),
         ("small_llama_N8", W.llama_1b2(world_size=8, layers=2, hidden=48, ffn=136, vocab=96)),
         # aligned plans for the flat kernel's general instance (N = 12 with pads, N = 1)
         ("small_llama_N12", W.llama_1b2(world_size=12, layers=1, hidden=96, ffn=104, vocab=100)),
         ("small_llama_N1", W.llama_1b2(world_size=1, layers=1, hidden=32, ffn=64, vocab=64)),
         # the largest world size the ABI takes (SS_MAX_WORLD), aligned: the
         # flat kernel with 8 ranks' loads in flight and the other 56 in a loop
         ("llama_N64", W.llama_1b2(world_size=64, layers=1, hidden=512, ffn=1024, vocab=128)),
         ("per_param_N12", W.ParamSet([f"p{i}" for i in range(4)], [(130, 3), (64,), (0, 4), (257, 8)],
                                      [4], 12, W.PER_PARAM_DIM0, torch.bfloat16, seed=11)),
         # 500 tiny aligned params: dozens of segment starts (and pad runs) in
         # every 2048-element block, so the flat kernel's binary search runs
         ("tiny_params_N4", W.ParamSet([f"t{i}" for i in range(500)],
                                       [(1 + (7 * i) % 9, 8) for i in range(500)],
                                       [500], 4, W.PER_PARAM_DIM0, torch.bfloat16, seed=13)),
         # 4.3M-8.9M params: more vectors than a small launch takes, so the
         # large forms of the N = 1, N = 16 and general instances run
         ("awkward1d_false_N1_large",
          W.awkward_1d(1, W.FLAT_ORIG_FALSE, torch.bfloat16, count=30, max_len=300_000)),
         ("awkward1d_false_N16_large",
          W.awkward_1d(16, W.FLAT_ORIG_FALSE, torch.bfloat16, count=30, max_len=300_000)),
         ("awkward1d_true_N17_large",
          W.awkward_1d(17, W.FLAT_ORIG_TRUE, torch.bfloat16, count=30, max_len=300_000)),
         ("llama_N1_large", W.llama_1b2(world_size=1, layers=2, hidden=512, ffn=1536, vocab=2048))]


def _state(ss, su):
    shards = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
    ss.fsdp_pack(su.plan, su.params, shards)
    master = torch.empty(su.total, device="cuda")
    m = torch.empty_like(master)
    v = torch.empty_like(master)
    ss.fsdp_init_master(su.plan, shards, master, m, v)
    return shards, master, m, v


@pytest.mark.parametrize("name,ps", CASES, ids=[c[0] for c in CASES])
def test_sharded_step_matches_two_calls_and_oracle(ss, name, ps):
    su = Setup(ss, ps)
    N, total, n = su.N, su.total, len(su.params)
    grads_cpu = W.make_rank_grads(ps)
    grads_params = [[g.cuda() for g in rank] for rank in grads_cpu]
    packed = []
    for r in range(N):
        b = torch.empty(total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, grads_params[r], b)
        packed.append(b)
    n_out = min(N, 3)
    # A: two calls
    sa, ma, mma, va = _state(ss, su)
    red_a = torch.zeros(total, device="cuda")
    outs_a = [torch.empty_like(p) for _ in range(n_out) for p in su.params]
    # B: one pass, packed gradients; C: one pass, per-parameter gradients
    sb, mb, mmb, vb = _state(ss, su)
    sc, mc, mmc, vc = _state(ss, su)
    red_b = torch.zeros(total, device="cuda")
    red_c = torch.zeros(total, device="cuda")
    outs_b, wholes = [], []
    for _ in range(n_out):
        for p in su.params:
            o, w = guarded(p.numel(), torch.bfloat16)
            outs_b.append(o)
            wholes.append(w)
    outs_c = [torch.empty_like(p) for _ in range(n_out) for p in su.params]
    flat_param_grads = [g for rank in grads_params for g in rank]
    torch.cuda.synchronize()
    for step in (1, 2):
        hp = ss.adamw_params(step=step, **_hp(step))
        ss.fsdp_reduce_scatter_adamw(su.plan, packed, ma, mma, va, sa, hp, red_a)
        ss.fsdp_all_gather_unpack(su.plan, sa, outs_a, n_out=n_out)
        ss.fsdp_sharded_step(su.plan, mb, mmb, vb, sb, hp, rank_grads=packed, params_out=outs_b,
                             n_out=n_out, reduced_grad_out=red_b)
        ss.fsdp_sharded_step(su.plan, mc, mmc, vc, sc, hp, rank_param_grads=flat_param_grads,
                             params_out=outs_c, n_out=n_out, reduced_grad_out=red_c)
        torch.cuda.synchronize()
        assert all(guards_intact(w) for w in wholes)
        np.testing.assert_array_equal(to_np(red_b).view(np.uint32), to_np(red_c).view(np.uint32))
        for x, y, z in ((sa, sb, sc), (ma, mb, mc), (mma, mmb, mmc), (va, vb, vc)):
            np.testing.assert_array_equal(to_np(x).view(np.uint8), to_np(y).view(np.uint8))
            np.testing.assert_array_equal(to_np(x).view(np.uint8), to_np(z).view(np.uint8))
        for x, y, z in zip(outs_a, outs_b, outs_c):
            np.testing.assert_array_equal(to_np(x), to_np(y))
            np.testing.assert_array_equal(to_np(x), to_np(z))
    # the reduced gradient on parameter elements equals the oracle's reduce-scatter
    ones = su.oracle_pack([np.full(p.numel(), 0x3F80, np.uint16) for p in su.params])
    data = ones != 0
    want = np.concatenate([oracle.reduce_scatter(N, g["shard_numel"],
                                                 [to_np(b)[g["base"]:g["base"] + N * g["shard_numel"]]
                                                  for b in packed]) for g in su.groups]) \
        if su.groups else np.zeros(0, np.float32)
    np.testing.assert_array_equal(to_np(red_b)[data], want[data])
    assert not to_np(red_b)[~data].any()          # pads never written


def test_sharded_step_windows_and_groups(ss):
    # N=7 per-parameter grads + 7 outputs: 14 pointers x 200 params > 2048, so the call
    # splits into parameter windows; group-by-group calls cover the plan in packed order
    ps = W.awkward_1d(7, W.FLAT_ORIG_FALSE, torch.bfloat16)
    ps.groups = [50, 0, 75, 75]
    su = Setup(ss, ps)
    N = su.N
    grads = [[g.cuda() for g in rank] for rank in W.make_rank_grads(ps)]
    flat = [g for rank in grads for g in rank]
    packed = []
    for r in range(N):
        b = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, grads[r], b)
        packed.append(b)
    results = []
    for mode in ("two_calls", "windows", "groups"):
        shards, master, m, v = _state(ss, su)
        outs = [torch.empty_like(p) for _ in range(N) for p in su.params]
        hp = ss.adamw_params(step=1)
        if mode == "two_calls":
            ss.fsdp_reduce_scatter_adamw(su.plan, packed, master, m, v, shards, hp)
            ss.fsdp_all_gather_unpack(su.plan, shards, outs, n_out=N)
        elif mode == "windows":
            ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp, rank_param_grads=flat,
                                 params_out=outs, n_out=N)
        else:
            for g in range(len(ps.groups)):
                ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp, rank_grads=packed,
                                     params_out=outs, n_out=N, group=g)
        torch.cuda.synchronize()
        results.append([to_np(t) for t in [shards, master, m, v] + outs])
    for other in results[1:]:
        for x, y in zip(results[0], other):
            np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("kind", [W.FLAT_ORIG_FALSE, W.FLAT_ORIG_TRUE, W.PER_PARAM_DIM0])
def test_sharded_step_groups_inside_one_vector(ss, kind):
    # one group per tiny parameter at N = 2: group ranges such as [10, 12) lie
    # inside one 8-element packed vector, others start or end mid-vector, so
    # the flat kernels' edge elements and their whole misaligned vectors both
    # run, with packed gradients and with the fused copy-in
    shapes = [(3,), (5,), (1,), (2,), (700,), (9,), (13,), (8,), (31,)]
    ps = W.ParamSet([f"q{i}" for i in range(len(shapes))], shapes, [1, 1, 1, 1, 1, 2, 1, 1], 2,
                    kind, torch.bfloat16, seed=17)
    su = Setup(ss, ps)
    N, n = su.N, len(su.params)
    grads = [[g.cuda() for g in rank] for rank in W.make_rank_grads(ps)]
    packed = []
    for r in range(N):
        b = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, grads[r], b)
        packed.append(b)
    # the same gradients as per-parameter views, each 2 * (r + i) mod 16 bytes
    # past a 16-byte boundary, for the fused copy-in
    views = []
    for r in range(N):
        for i, g in enumerate(grads[r]):
            o, _ = guarded(g.numel() + 8, torch.bfloat16)
            v = o[(r + i) % 8:(r + i) % 8 + g.numel()]
            v.copy_(g.view(-1))
            views.append(v)
    results, wholes, firsts = [], [], []
    for mode in ("two_calls", "one_pass", "copy_in"):
        shards, master, m, v = _state(ss, su)
        red = torch.zeros(su.total, device="cuda")
        outs = []
        for _ in range(2):
            for p in su.params:
                o, w = guarded(p.numel() + 1, torch.bfloat16)
                outs.append(o[1:])          # 2 bytes past a 16-byte boundary
                wholes.append(w)
                firsts.append(o[:1])        # the element before: never written
        for step in (1, 2):
            hp = ss.adamw_params(step=step, **_hp(step))
            for g in range(len(ps.groups)):
                if mode == "two_calls":
                    ss.fsdp_reduce_scatter_adamw(su.plan, packed, master, m, v, shards, hp, red,
                                                 group=g)
                    ss.fsdp_all_gather_unpack(su.plan, shards, outs, n_out=2, group=g)
                elif mode == "one_pass":
                    ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp, rank_grads=packed,
                                         params_out=outs, n_out=2, reduced_grad_out=red, group=g)
                else:
                    ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp, rank_param_grads=views,
                                         params_out=outs, n_out=2, reduced_grad_out=red, group=g)
        torch.cuda.synchronize()
        results.append([to_np(t) for t in [shards, master, m, v, red] + outs])
    assert all(guards_intact(w) for w in wholes)
    assert all(int(to_np(f).view(np.uint16)[0]) == SENTINEL_BF16 for f in firsts)
    for other in results[1:]:
        for x, y in zip(results[0], other):
            np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))
    for j in range(2):
        for i in range(n):
            assert results[1][5 + j * n + i].size == su.params[i].numel()


def test_prepared_step_equals_the_call(ss):
    # ss.ShardedStep marshals the arguments once; its steps must be the plain
    # call's, bit for bit, for packed and per-parameter gradients
    ps = W.llama_1b2(world_size=4, layers=2, hidden=48, ffn=136, vocab=96)
    su = Setup(ss, ps)
    N = su.N
    grads = [[g.cuda() for g in rank] for rank in W.make_rank_grads(ps)]
    flat = [g for rank in grads for g in rank]
    packed = []
    for r in range(N):
        b = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, grads[r], b)
        packed.append(b)
    for src in ("packed", "per_param"):
        kw = {"rank_grads": packed} if src == "packed" else {"rank_param_grads": flat}
        sa, ma, mma, va = _state(ss, su)
        sb, mb, mmb, vb = _state(ss, su)
        outs_a = [torch.empty_like(p) for p in su.params]
        outs_b = [torch.empty_like(p) for p in su.params]
        call = ss.ShardedStep(su.plan, mb, mmb, vb, sb, ss.adamw_params(step=1, **_hp(1)),
                              params_out=outs_b, n_out=1, **kw)
        for step in (1, 2, 3):
            ss.fsdp_sharded_step(su.plan, ma, mma, va, sa, ss.adamw_params(step=step, **_hp(1)),
                                 params_out=outs_a, n_out=1, **kw)
            call(step)
        torch.cuda.synchronize()
        for x, y in zip([sa, ma, mma, va] + outs_a, [sb, mb, mmb, vb] + outs_b):
            np.testing.assert_array_equal(to_np(x).view(np.uint8), to_np(y).view(np.uint8))
    with pytest.raises(ss.ShardStateError):
        ss.ShardedStep(su.plan, mb, mmb, vb, sb, ss.adamw_params(step=1, **_hp(1)),
                       rank_grads=packed, params_out=outs_b, n_out=1)(0)  # step 0: EINVAL


def test_small_launches_between_dependent_work(ss):
    """The small one-pass form lets the next launch on the stream start early
    and waits for its predecessor before touching memory.  Here every step's
    gradients are made by torch kernels from the previous step's gathered
    parameters, with no synchronisation anywhere, so each step kernel sits
    between kernels that produce its inputs and consume its outputs; four
    steps of that chain equal, bit for bit, the same chain through the
    two-call path (pack, RS+AdamW, all-gather: launches without early start)."""
    ps = W.tiny_mlp(2, W.FLAT_ORIG_TRUE)
    su = Setup(ss, ps)
    N = su.N
    results = []
    for mode in ("two_calls", "one_pass"):
        shards, master, m, v = _state(ss, su)
        outs = [p.clone() for p in su.params]
        packed = [torch.empty(su.total, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
        torch.cuda.synchronize()
        for step in (1, 2, 3, 4):
            # rank r's gradient of each parameter, from the gathered parameters
            grads = [[(o.float() * (0.01 * (r + 1)) - 1e-3 * step).to(torch.bfloat16) for o in outs]
                     for r in range(N)]
            hp = ss.adamw_params(step=step, **_hp(step))
            if mode == "two_calls":
                for r in range(N):
                    ss.fsdp_pack(su.plan, grads[r], packed[r])
                ss.fsdp_reduce_scatter_adamw(su.plan, packed, master, m, v, shards, hp)
                ss.fsdp_all_gather_unpack(su.plan, shards, outs)
            else:
                ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp,
                                     rank_param_grads=[g for rank in grads for g in rank],
                                     params_out=outs, n_out=1)
        torch.cuda.synchronize()
        results.append([to_np(t) for t in [shards, master, m, v] + outs])
    for x, y in zip(*results):
        np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))


ORACLE_STATE_CASES = [
    ("small_llama_N8", W.llama_1b2(world_size=8, layers=2, hidden=48, ffn=136, vocab=96)),
    ("awkward1d_false_N7", W.awkward_1d(7, W.FLAT_ORIG_FALSE, torch.bfloat16, count=80)),
    ("awkward1d_false_N17", W.awkward_1d(17, W.FLAT_ORIG_FALSE, torch.bfloat16, count=60)),
    ("awkward1d_true_N24", W.awkward_1d(24, W.FLAT_ORIG_TRUE, torch.bfloat16, count=60))]


@pytest.mark.parametrize("name,ps", ORACLE_STATE_CASES, ids=[c[0] for c in ORACLE_STATE_CASES])
def test_sharded_step_state_against_oracle(ss, name, ps):
    """The fused copy-in (per-parameter gradients) against the oracle over
    three steps: aligned (N = 8) and misaligned runs (N = 7, 17, 24)."""
    su = Setup(ss, ps)
    N, total = su.N, su.total
    shards, master, m, v = _state(ss, su)
    grads_cpu = W.make_rank_grads(ps)
    flat = [g.cuda() for rank in grads_cpu for g in rank]
    packed_np = [su.oracle_pack([to_np(g) for g in rank]) for rank in grads_cpu]
    outs = [torch.empty_like(p) for p in su.params]
    for step in (1, 2, 3):
        pm, pmm, pv = to_np(master), to_np(m), to_np(v)
        ss.fsdp_sharded_step(su.plan, master, m, v, shards, ss.adamw_params(step=step, **_hp(step)),
                             rank_param_grads=flat, params_out=outs, n_out=1)
        torch.cuda.synchronize()
        om, omm, ov = pm.copy(), pmm.copy(), pv.copy()
        o_params, o_red = oracle.reduce_scatter_adamw(N, su.info.shard_numel, packed_np, om, omm, ov,
                                                      step=step, **_hp(step))
        check_adamw_state(to_np(master), to_np(m), to_np(v), om, omm, ov, pm, pmm, o_red)
        check_bf16_params(to_np(shards), o_params, to_np(master), om, pm)
        want = su.oracle_unpack(to_np(shards))[0]
        for o, w in zip(outs, want):
            np.testing.assert_array_equal(to_np(o), w)


def test_sharded_step_full_size_equals_two_calls(ss):
    ps = W.llama_1b2()
    su = Setup(ss, ps, make_values=False)
    total, N = su.total, su.N
    gen = torch.Generator(device="cuda").manual_seed(4)
    init = (torch.randn(total, device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
    grads = W.make_packed_rank_grads(N, total, 1e-3, 4, device="cuda")
    res = []
    for mode in ("two_calls", "one_pass"):
        shards = init.clone()
        master = torch.empty(total, device="cuda")
        m = torch.empty_like(master)
        v = torch.empty_like(master)
        ss.fsdp_init_master(su.plan, shards, master, m, v)
        outs = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in ps.shapes]
        for step in (1, 2):
            hp = ss.adamw_params(step=step)
            if mode == "two_calls":
                ss.fsdp_reduce_scatter_adamw(su.plan, grads, master, m, v, shards, hp)
                ss.fsdp_all_gather_unpack(su.plan, shards, outs)
            else:
                ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp, rank_grads=grads,
                                     params_out=outs, n_out=1)
        torch.cuda.synchronize()
        res.append((shards, master, m, v, outs))
    a, b = res
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    for x, y in zip(a[1:4], b[1:4]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    for x, y in zip(a[4], b[4]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    del res, a, b, grads
    torch.cuda.empty_cache()


def _per_param_places(su, idx: np.ndarray):
    """Parameter and element index of packed elements idx (sorted) of a
    PER_PARAM_DIM0 plan, from the oracle's layout of each group: rank r's chunk
    of parameter i holds rows r*c_i .. r*c_i + c_i - 1 from shard offset off_i
    on ("FSDP1 vs FSDP2", section 03: FSDP2's per-parameter dim-0 chunks).
    Returns (param, k), param -1 for a pad element."""
    assert su.kind == W.PER_PARAM_DIM0
    param = np.full(idx.size, -1, np.int64)
    k = np.zeros(idx.size, np.int64)
    for g, grp in enumerate(su.groups):
        a, b, d0, inner = su._group_args(g)
        lay = oracle.layout(su.kind, su.N, 2, d0, inner)
        S = lay["shard_numel"]
        lo, hi = np.searchsorted(idx, [grp["base"], grp["base"] + su.N * S])
        rel = idx[lo:hi] - grp["base"]
        r, local = rel // S, rel % S
        off = np.asarray(lay["offsets"], np.int64)
        rows = np.asarray(lay["chunk_rows"], np.int64)
        inn = np.asarray(inner, np.int64)
        d0 = np.asarray(d0, np.int64)
        i = np.searchsorted(off, local, side="right") - 1
        # empty parameters share their offset with the next one: take the
        # last parameter starting at or before `local` that holds elements
        j = local - off[i]
        row = r * rows[i] + j // np.maximum(inn[i], 1)
        inside = (j < rows[i] * inn[i]) & (row < d0[i])
        param[lo:hi] = np.where(inside, a + i, -1)
        k[lo:hi] = np.where(inside, row * inn[i] + j % np.maximum(inn[i], 1), 0)
    return param, k


def test_headline_step_full_size_against_the_oracle(ss):
    """The launch the benchmark times -- fsdp_sharded_step over the whole
    1.2B-shaped model (N = 8, packed gradients, n_out = 1) -- checked against
    the oracle in one test, over two steps: on 2M sampled packed elements the
    reduce-scatter + AdamW state and bf16 shard against
    oracle.reduce_scatter_adamw applied to the sampled inputs ("Scaling data
    parallel", sections 9.1-9.3: reduce-scatter, then AdamW on each rank's own
    shard in fp32, then the cast), and the unpacked output of every sampled
    data element against the same bf16 value ("FSDP1 vs FSDP2", section 04:
    the group all-gather returns every parameter whole)."""
    ps = W.llama_1b2()
    su = Setup(ss, ps, make_values=False)
    total, N = su.total, su.N
    assert total == 1_364_297_728 and N == 8
    gen = torch.Generator(device="cuda").manual_seed(4)
    shards = (torch.randn(total, device="cuda", generator=gen) * ps.param_std).to(torch.bfloat16)
    master = torch.empty(total, device="cuda")
    m = torch.empty_like(master)
    v = torch.empty_like(master)
    ss.fsdp_init_master(su.plan, shards, master, m, v)
    grads = W.make_packed_rank_grads(N, total, ps.grad_std, ps.seed, device="cuda")
    outs = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in ps.shapes]
    sgen = torch.Generator(device="cuda").manual_seed(4242)
    idx_t = torch.unique(torch.randint(0, total, (1 << 21,), device="cuda", generator=sgen))
    idx_t = idx_t[:idx_t.numel() // N * N]
    idx = idx_t.cpu().numpy()
    param, k = _per_param_places(su, idx)
    data = param >= 0
    assert data.all()  # every dim0 of this model divides by 8: no pads
    for step in (1, 2):
        in_master = master[idx_t].cpu().numpy()
        in_m = m[idx_t].cpu().numpy()
        in_v = v[idx_t].cpu().numpy()
        in_g = [to_np(gr[idx_t]) for gr in grads]
        launches = ss.ss_launch_count()
        ss.fsdp_sharded_step(su.plan, master, m, v, shards, ss.adamw_params(step=step, **_hp(step)),
                             rank_grads=grads, params_out=outs, n_out=1)
        torch.cuda.synchronize()
        assert ss.ss_launch_count() - launches == 1  # the one flat launch
        om, omm, ov = in_master.copy(), in_m.copy(), in_v.copy()
        o_params, o_red = oracle.reduce_scatter_adamw(N, idx.size // N, in_g, om, omm, ov,
                                                      step=step, **_hp(step))
        g_master = master[idx_t].cpu().numpy()
        check_adamw_state(g_master, m[idx_t].cpu().numpy(), v[idx_t].cpu().numpy(), om, omm, ov,
                          in_master, in_m, o_red)
        g_shard = to_np(shards[idx_t])
        check_bf16_params(g_shard, o_params, g_master, om, in_master)
        # the unpacked outputs hold the same bf16 values, parameter by parameter
        got = np.empty(idx.size, np.uint16)
        for i in np.unique(param):
            sel = np.nonzero(param == i)[0]
            flat = outs[i].reshape(-1)
            assert k[sel].min() >= 0 and k[sel].max() < flat.numel()  # checked on the host
            got[sel] = to_np(flat[torch.from_numpy(k[sel]).to("cuda")])
        np.testing.assert_array_equal(got, g_shard)
    del grads, outs
    torch.cuda.empty_cache()


def test_sharded_step_full_size_copy_in_equals_pack_and_two_calls(ss):
    """The 1.2B model with the gradients as 8 per-parameter sets (fused
    copy-in, the flat kernel's UNPACKED form): bit-identical to packing each
    set and running RS+AdamW + all-gather."""
    ps = W.llama_1b2()
    su = Setup(ss, ps, make_values=False)
    total, N = su.total, su.N
    gen = torch.Generator(device="cuda").manual_seed(44)
    init = (torch.randn(total, device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
    sets = [[(torch.randn(s, device="cuda", generator=gen) * 1e-3).to(torch.bfloat16)
             for s in ps.shapes] for _ in range(N)]
    flat_sets = [g for rank in sets for g in rank]
    res = []
    for mode in ("pack_two_calls", "copy_in"):
        shards = init.clone()
        master = torch.empty(total, device="cuda")
        m = torch.empty_like(master)
        v = torch.empty_like(master)
        ss.fsdp_init_master(su.plan, shards, master, m, v)
        outs = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in ps.shapes]
        hp = ss.adamw_params(step=1)
        if mode == "pack_two_calls":
            packed = []
            for r in range(N):
                b = torch.empty(total, dtype=torch.bfloat16, device="cuda")
                ss.fsdp_pack(su.plan, sets[r], b)
                packed.append(b)
            ss.fsdp_reduce_scatter_adamw(su.plan, packed, master, m, v, shards, hp)
            ss.fsdp_all_gather_unpack(su.plan, shards, outs)
            torch.cuda.synchronize()
            del packed
        else:
            ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp, rank_param_grads=flat_sets,
                                 params_out=outs, n_out=1)
            torch.cuda.synchronize()
        res.append((shards, master, m, v, outs))
    a, b = res
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    for x, y in zip(a[1:4], b[1:4]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    for x, y in zip(a[4], b[4]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    del res, a, b, sets, flat_sets
    torch.cuda.empty_cache()


LARGE_COPY_IN_CASES = [
    ("awkward1d_false_N9_80M",
     lambda: W.awkward_1d(9, W.FLAT_ORIG_FALSE, torch.bfloat16, count=40, max_len=4_500_000)),
    ("awkward2d_N7_67M", lambda: W.awkward_2d(7, count=200, max_rows=200_000)),
    # 800 parameters in one group: 8 pointers each overflow the 2048-slot
    # table, so the call runs in parameter windows, each window's data in 7
    # runs (one per rank shard): 28 launches, chained by programmatic
    # dependent launch
    ("awkward2d_N7_800params_windows", lambda: W.awkward_2d(7, count=800, max_rows=40_000)),
]


@pytest.mark.parametrize("name,make", LARGE_COPY_IN_CASES, ids=[c[0] for c in LARGE_COPY_IN_CASES])
def test_sharded_step_large_copy_in_equals_pack_and_two_calls(ss, name, make):
    """Per-parameter gradients on misaligned plans of 67M-87M params (N = 9:
    the general instance, ranks in two batches; N = 7 PER_PARAM_DIM0: its own
    instance, with pads in most rank chunks): tens of waves of warps of 8
    rounds each, and the step must equal packing each set and running the
    two calls bit for bit (pads, zero in the packed shards, stay zero)."""
    ps = make()
    su = Setup(ss, ps, make_values=False)
    total, N = su.total, su.N
    assert total >= 30_000_000
    gen = torch.Generator(device="cuda").manual_seed(45)
    # shards packed from parameters, so the pads hold zero as the step expects
    init = torch.empty(total, dtype=torch.bfloat16, device="cuda")
    ss.fsdp_pack(su.plan, [(torch.randn(s, device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
                           for s in ps.shapes], init)
    sets = [[(torch.randn(s, device="cuda", generator=gen) * 1e-3).to(torch.bfloat16)
             for s in ps.shapes] for _ in range(N)]
    res = []
    for mode in ("pack_two_calls", "copy_in"):
        shards = init.clone()
        master = torch.empty(total, device="cuda")
        m = torch.empty_like(master)
        v = torch.empty_like(master)
        ss.fsdp_init_master(su.plan, shards, master, m, v)
        outs = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in ps.shapes]
        hp = ss.adamw_params(step=1)
        if mode == "pack_two_calls":
            packed = []
            for r in range(N):
                b = torch.empty(total, dtype=torch.bfloat16, device="cuda")
                ss.fsdp_pack(su.plan, sets[r], b)
                packed.append(b)
            ss.fsdp_reduce_scatter_adamw(su.plan, packed, master, m, v, shards, hp)
            ss.fsdp_all_gather_unpack(su.plan, shards, outs)
            torch.cuda.synchronize()
            del packed
        else:
            ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp,
                                 rank_param_grads=[g for rank in sets for g in rank],
                                 params_out=outs, n_out=1)
            torch.cuda.synchronize()
        res.append((shards, master, m, v, outs))
    a, b = res
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    for x, y in zip(a[1:4], b[1:4]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    for x, y in zip(a[4], b[4]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    del res, a, b, sets
    torch.cuda.empty_cache()


def test_sharded_step_argument_errors(ss):
    su = Setup(ss, W.tiny_mlp())
    shards, master, m, v = _state(ss, su)
    g = [torch.empty(su.total, dtype=torch.bfloat16, device="cuda")] * 2
    hp = ss.adamw_params()
    with pytest.raises(ss.ShardStateError) as e:   # neither gradient source
        ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp)
    assert e.value.status == ss.SS_EINVAL
    with pytest.raises(ss.ShardStateError) as e:   # both
        ss.fsdp_sharded_step(su.plan, master, m, v, shards, hp, rank_grads=g,
                             rank_param_grads=[p for p in su.params] * 2)
    assert e.value.status == ss.SS_EINVAL
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_sharded_step(su.plan, master[1:], m, v, shards, hp, rank_grads=g)
    assert e.value.status == ss.SS_EALIGN
    f32plan = ss.fsdp_plan_create(ss.SS_FLAT_ORIG_TRUE, 2, 4, [16])
    with pytest.raises(ss.ShardStateError) as e:
        ss.fsdp_sharded_step(f32plan, master, m, v, master, hp, rank_grads=[master, master])
    assert e.value.status == ss.SS_EINVAL
    torch.cuda.synchronize()


def test_zero12_step_every_rank_gets_the_parameters(ss):
    """The ZeRO-1/2 step ("Scaling data parallel" 9.1-9.2): RS+AdamW, then the
    updated bf16 parameters all-gathered to every one of the N ranks.  The one
    pass with n_out = N must equal RS+AdamW followed by the all-gather with
    n_out = N bit for bit, and every replica must equal the oracle's unpack of
    the new shards."""
    ps = W.llama_1b2(world_size=8, layers=2, hidden=48, ffn=136, vocab=96)
    su = Setup(ss, ps)
    N, total = su.N, su.total
    grads_cpu = W.make_rank_grads(ps)
    packed = []
    for r in range(N):
        b = torch.empty(total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, [g.cuda() for g in grads_cpu[r]], b)
        packed.append(b)
    sa, ma, mma, va = _state(ss, su)
    sb, mb, mmb, vb = _state(ss, su)
    outs_a = [torch.empty_like(p) for _ in range(N) for p in su.params]
    outs_b, wholes = [], []
    for _ in range(N):
        for p in su.params:
            o, w = guarded(p.numel(), torch.bfloat16)
            outs_b.append(o)
            wholes.append(w)
    for step in (1, 2):
        hp = ss.adamw_params(step=step, **_hp(step))
        ss.fsdp_reduce_scatter_adamw(su.plan, packed, ma, mma, va, sa, hp)
        ss.fsdp_all_gather_unpack(su.plan, sa, outs_a, n_out=N)
        ss.fsdp_sharded_step(su.plan, mb, mmb, vb, sb, hp, rank_grads=packed, params_out=outs_b,
                             n_out=N)
        torch.cuda.synchronize()
        for x, y in ((sa, sb), (ma, mb), (mma, mmb), (va, vb)):
            np.testing.assert_array_equal(to_np(x).view(np.uint8), to_np(y).view(np.uint8))
        want = su.oracle_unpack(to_np(sb), n_out=N)
        n = len(su.params)
        for j in range(N):
            for i in range(n):
                np.testing.assert_array_equal(to_np(outs_a[j * n + i]), to_np(outs_b[j * n + i]))
                np.testing.assert_array_equal(to_np(outs_b[j * n + i]), want[j][i])
    assert all(guards_intact(w) for w in wholes)


def test_sharded_step_max_replicas(ss):
    """n_out = SS_MAX_REPLICAS outputs from the one pass equal the all-gather
    with the same replica count after RS+AdamW, bit for bit."""
    ps = W.tiny_mlp(2, W.FLAT_ORIG_TRUE)
    su = Setup(ss, ps)
    N, total, R = su.N, su.total, ss.SS_MAX_REPLICAS
    packed = []
    for r, rank in enumerate(W.make_rank_grads(ps)):
        b = torch.empty(total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, [g.cuda() for g in rank], b)
        packed.append(b)
    sa, ma, mma, va = _state(ss, su)
    sb, mb, mmb, vb = _state(ss, su)
    outs_a = [torch.empty_like(p) for _ in range(R) for p in su.params]
    outs_b = [torch.empty_like(p) for _ in range(R) for p in su.params]
    hp = ss.adamw_params(step=1, **_hp(1))
    ss.fsdp_reduce_scatter_adamw(su.plan, packed, ma, mma, va, sa, hp)
    ss.fsdp_all_gather_unpack(su.plan, sa, outs_a, n_out=R)
    ss.fsdp_sharded_step(su.plan, mb, mmb, vb, sb, hp, rank_grads=packed, params_out=outs_b, n_out=R)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(sa), to_np(sb))
    for x, y in zip(outs_a, outs_b):
        np.testing.assert_array_equal(to_np(x), to_np(y))
