"""Per-parameter tensors at every 2-byte offset modulo 16 bytes.

A framework hands the library views into larger allocations, so a parameter's
data pointer is only guaranteed to be element aligned.  Each parameter here
sits at its own offset of 0..7 bf16 elements into a guarded buffer; the pack,
the all-gather + unpack and the one-pass step must give bit-identical results
to the same calls on 16-byte aligned tensors (and the pack the oracle's), and
must not write a byte outside each view.  On a plan whose runs are all whole
16-byte vectors this drives the general (realigning) kernels that the aligned
fast paths otherwise hide.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_common import Setup
from tests.helpers import to_np

pytestmark = pytest.mark.gpu

SENT = 0x7FA1  # a NaN pattern no kernel writes


@pytest.fixture(scope="module")
def ss():
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    return ss


def _shifted(numel, shift):
    """(view at `shift` elements into a sentinel-filled buffer, whole buffer)."""
    whole = torch.empty(numel + 16, dtype=torch.bfloat16, device="cuda")
    whole.view(torch.int16).fill_(SENT)
    return whole[shift:shift + numel], whole


def _outside_intact(whole, shift, numel):
    w = to_np(whole).view(np.uint16)
    return bool((w[:shift] == SENT).all() and (w[shift + numel:] == SENT).all())


CASES = [("small_llama_N8", W.llama_1b2(world_size=8, layers=2, hidden=48, ffn=136, vocab=96)),
         ("awkward1d_false_N7", W.awkward_1d(7, W.FLAT_ORIG_FALSE, torch.bfloat16)),
         ("awkward2d_N3", W.awkward_2d(3))]


@pytest.mark.parametrize("name,ps", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("base", [1, 2, 4])
def test_pack_and_all_gather_at_any_offset(ss, name, ps, base):
    su = Setup(ss, ps)
    numels = [p.numel() for p in su.params]
    shifts = [(base + 3 * i) % 8 for i in range(len(numels))]
    views, wholes = [], []
    for p, s in zip(su.params, shifts):
        v, w = _shifted(p.numel(), s)
        v.copy_(p.view(-1))
        views.append(v)
        wholes.append(w)
    ref = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
    got = torch.empty_like(ref)
    ss.fsdp_pack(su.plan, [p.view(-1) for p in su.params], ref)
    ss.fsdp_pack(su.plan, views, got)
    torch.cuda.synchronize()
    want = su.oracle_pack(su.params_np())
    np.testing.assert_array_equal(to_np(got), want)
    np.testing.assert_array_equal(to_np(ref), want)
    # all-gather from the packed shards into shifted outputs, two replicas
    outs, out_wholes = [], []
    for _ in range(2):
        for n, s in zip(numels, shifts):
            v, w = _shifted(n, (s + 5) % 8)
            outs.append(v)
            out_wholes.append(w)
    ss.fsdp_all_gather_unpack(su.plan, got, outs, n_out=2)
    torch.cuda.synchronize()
    for j in range(2):
        for i, p in enumerate(su.params_cpu):
            np.testing.assert_array_equal(to_np(outs[j * len(numels) + i]), to_np(p))
    for v, w, n in zip(outs, out_wholes, numels * 2):
        assert _outside_intact(w, (v.data_ptr() - w.data_ptr()) // 2, n)


@pytest.mark.parametrize("name,ps", CASES, ids=[c[0] for c in CASES])
def test_sharded_step_at_any_offset(ss, name, ps):
    su = Setup(ss, ps)
    N, n = su.N, len(su.params)
    grads_cpu = W.make_rank_grads(ps)
    aligned_grads = [g.cuda().view(-1) for rank in grads_cpu for g in rank]
    shifted_grads = []
    for idx, g in enumerate(aligned_grads):
        v, _ = _shifted(g.numel(), (idx * 5 + 1) % 8)
        v.copy_(g)
        shifted_grads.append(v)
    numels = [p.numel() for p in su.params]

    def state():
        shards = torch.empty(su.total, dtype=torch.bfloat16, device="cuda")
        ss.fsdp_pack(su.plan, su.params, shards)
        master = torch.empty(su.total, device="cuda")
        m, v = torch.empty_like(master), torch.empty_like(master)
        ss.fsdp_init_master(su.plan, shards, master, m, v)
        return shards, master, m, v

    sa, ma, mma, va = state()
    sb, mb, mmb, vb = state()
    outs_a = [torch.empty(k, dtype=torch.bfloat16, device="cuda") for k in numels]
    outs_b, wholes = [], []
    for i, k in enumerate(numels):
        v, w = _shifted(k, (7 * i + 3) % 8)
        outs_b.append(v)
        wholes.append(w)
    for step in (1, 2):
        hp = ss.adamw_params(step=step, **{k: W.adamw_hparams(step)[k]
                                            for k in ("lr", "beta1", "beta2", "eps", "weight_decay")})
        ss.fsdp_sharded_step(su.plan, ma, mma, va, sa, hp, rank_param_grads=aligned_grads,
                             params_out=outs_a, n_out=1)
        ss.fsdp_sharded_step(su.plan, mb, mmb, vb, sb, hp, rank_param_grads=shifted_grads,
                             params_out=outs_b, n_out=1)
        torch.cuda.synchronize()
        for x, y in ((sa, sb), (ma, mb), (mma, mmb), (va, vb)):
            np.testing.assert_array_equal(to_np(x).view(np.uint8), to_np(y).view(np.uint8))
        for x, y in zip(outs_a, outs_b):
            np.testing.assert_array_equal(to_np(x), to_np(y))
    for v, w, k in zip(outs_b, wholes, numels):
        assert _outside_intact(w, (v.data_ptr() - w.data_ptr()) // 2, k)
    assert N * n == len(shifted_grads)
