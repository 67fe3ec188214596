"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one oracle function to something the pages or mathematics fix:
printed worked examples and ledger tables (tests/golden/), library routines
that realise the same definition (torch.chunk, torch.optim.AdamW, torch's
bf16 cast, torch.autograd), closed forms, invariants and brute force.
"""
import itertools
import os
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import dp_equivalence, ledger
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KIND = {"flat_orig_false": oracle.FLAT_ORIG_FALSE, "flat_orig_true": oracle.FLAT_ORIG_TRUE,
        "per_param_dim0": oracle.PER_PARAM_DIM0}


def _bits(t: torch.Tensor) -> np.ndarray:
    """torch bf16/fp32 tensor -> numpy uint16 / float32 (same bytes)."""
    t = t.contiguous().reshape(-1)
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().astype(np.float32, copy=True)


def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


# ---------------------------------------------------------------------------
# layout
# ---------------------------------------------------------------------------

def test_worked_example_3_5():
    rows = list(_golden_rows("worked_example_3_5.txt"))
    assert len(rows) == 3
    for name, N, eb, numels, per_rank, total, offs, crows in rows:
        numels = [int(x) for x in numels.split(",")]
        lay = oracle.layout(KIND[name], int(N), int(eb), numels)
        assert lay["shard_numel"] == int(per_rank), name
        assert lay["total_numel"] == int(total), name
        assert lay["offsets"] == [int(x) for x in offs.split(",")], name
        assert lay["chunk_rows"] == [int(x) for x in crows.split(",")], name
    # the page's relative statements: FSDP2 = 1.5x FSDP1 default, 0.75x use_orig_params=True
    ff = oracle.layout(oracle.FLAT_ORIG_FALSE, 4, 2, [3, 5])["shard_numel"]
    ft = oracle.layout(oracle.FLAT_ORIG_TRUE, 4, 2, [3, 5])["shard_numel"]
    pp = oracle.layout(oracle.PER_PARAM_DIM0, 4, 2, [3, 5])["shard_numel"]
    assert pp == 1.5 * ff and pp == 0.75 * ft


def _torch_chunk_flat(values, N):
    """FSDP1 default: torch.flatten(cat).chunk(N), each chunk padded to chunks[0].numel(),
    ranks without a chunk get an all-pad chunk."""
    flat = torch.cat([v.reshape(-1) for v in values]) if values else torch.zeros(0)
    chunks = list(torch.flatten(flat).chunk(N)) if flat.numel() else []
    c = chunks[0].numel() if chunks else 0
    out = []
    for r in range(N):
        piece = chunks[r] if r < len(chunks) else flat[:0]
        pad = torch.zeros(c - piece.numel(), dtype=flat.dtype)
        out.append(torch.cat([piece, pad]))
    return torch.cat(out) if out else flat[:0], c


def _bf16_vals(numels, seed):
    g = torch.Generator().manual_seed(seed)
    return [(torch.rand(n, generator=g) * 2 - 1).to(torch.bfloat16) for n in numels]


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8])
def test_flat_orig_false_is_torch_chunk(N):
    rng = random.Random(N)
    for trial in range(6):
        numels = [rng.randint(0, 40) for _ in range(rng.randint(0, 7))]
        vals = _bf16_vals(numels, trial)
        expect, c = _torch_chunk_flat(vals, N)
        lay = oracle.layout(oracle.FLAT_ORIG_FALSE, N, 2, numels)
        assert lay["shard_numel"] == c
        got = oracle.pack(oracle.FLAT_ORIG_FALSE, N, 2, numels, None, [_bits(v) for v in vals])
        np.testing.assert_array_equal(got, _bits(expect))


@pytest.mark.parametrize("N", [3, 5, 7])
def test_flat_orig_false_awkward_config(N):
    ps = W.awkward_1d(N, W.FLAT_ORIG_FALSE, torch.bfloat16)
    vals = [v.reshape(-1) for v in W.make_params(ps)]
    expect, c = _torch_chunk_flat(vals, N)
    got = oracle.pack(oracle.FLAT_ORIG_FALSE, N, 2, ps.numels(), None, [_bits(v) for v in vals])
    np.testing.assert_array_equal(got, _bits(expect))


def _torch_chunk_per_param(values, dim0, inner, N):
    """FSDP2: each param chunked on dim 0 with torch.chunk, padded to ceil(d0/N) rows,
    missing chunks empty; rank r's shard concatenates its chunk of every param."""
    ranks = [[] for _ in range(N)]
    for v, d0, inn in zip(values, dim0, inner):
        v2 = v.reshape(d0, inn)
        chunks = list(torch.chunk(v2, N, dim=0)) if d0 > 0 else []
        rows = chunks[0].shape[0] if chunks else 0
        for r in range(N):
            piece = chunks[r] if r < len(chunks) else v2[:0]
            pad = torch.zeros((rows - piece.shape[0], inn), dtype=v.dtype)
            ranks[r].append(torch.cat([piece, pad]).reshape(-1))
    return torch.cat([torch.cat(x) if x else torch.zeros(0, dtype=torch.bfloat16) for x in ranks])


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8])
def test_per_param_is_torch_chunk_dim0(N):
    rng = random.Random(100 + N)
    for trial in range(6):
        n = rng.randint(0, 7)
        dim0 = [rng.randint(0, 23) for _ in range(n)]
        inner = [rng.choice([1, 2, 3, 8]) for _ in range(n)]
        vals = _bf16_vals([d * i for d, i in zip(dim0, inner)], 50 + trial)
        expect = _torch_chunk_per_param(vals, dim0, inner, N)
        got = oracle.pack(oracle.PER_PARAM_DIM0, N, 2, dim0, inner, [_bits(v) for v in vals])
        np.testing.assert_array_equal(got, _bits(expect))


def test_per_param_awkward_2d_config():
    for N in (3, 5, 7):
        ps = W.awkward_2d(N)
        d0, inner = ps.dim0_inner()
        vals = [v.reshape(-1) for v in W.make_params(ps)]
        expect = _torch_chunk_per_param(vals, d0, inner, N)
        got = oracle.pack(oracle.PER_PARAM_DIM0, N, 2, d0, inner, [_bits(v) for v in vals])
        np.testing.assert_array_equal(got, _bits(expect))


def _byte_slot_simulation(numels, N, elem_bytes):
    """FSDP1 use_orig_params=True by byte addresses: the first param starts at byte 0;
    every later param starts at the first byte address >= the previous end that a
    16-byte boundary allows; the buffer is then extended until its element count is
    a multiple of N."""
    addr = 0
    starts = []
    for i, n in enumerate(numels):
        if i > 0:
            addr = -(-addr // 16) * 16
        starts.append(addr // elem_bytes)
        addr += n * elem_bytes
    count = addr // elem_bytes
    while count % N:
        count += 1
    return starts, count // N


@pytest.mark.parametrize("elem_bytes", [2, 4])
def test_flat_orig_true_brute_force(elem_bytes):
    a = 16 // elem_bytes
    for N in range(1, 9):
        for sizes in itertools.product(range(0, 11), repeat=3):
            lay = oracle.layout(oracle.FLAT_ORIG_TRUE, N, elem_bytes, list(sizes))
            starts, c = _byte_slot_simulation(sizes, N, elem_bytes)
            assert lay["offsets"] == starts
            assert lay["shard_numel"] == c
            offs = lay["offsets"]
            for i in range(1, 3):
                pad = offs[i] - (offs[i - 1] + sizes[i - 1])
                assert 0 <= pad <= a - 1 and offs[i] % a == 0
            assert lay["total_numel"] % N == 0


def test_flat_orig_true_pack_is_padded_flat_chunked():
    """use_orig_params=True: flat = [p0, pad, p1, pad, ...] + world pad; torch.chunk(N)
    then yields N equal chunks, which are the rank shards side by side."""
    for N in (3, 5, 7):
        ps = W.awkward_1d(N, W.FLAT_ORIG_TRUE, torch.bfloat16)
        vals = [v.reshape(-1) for v in W.make_params(ps)]
        lay = oracle.layout(oracle.FLAT_ORIG_TRUE, N, 2, ps.numels())
        pieces, pos = [], 0
        for off, v in zip(lay["offsets"], vals):
            pieces.append(torch.zeros(off - pos, dtype=torch.bfloat16))
            pieces.append(v)
            pos = off + v.numel()
        pieces.append(torch.zeros(lay["total_numel"] - pos, dtype=torch.bfloat16))
        flat = torch.cat(pieces)
        chunks = flat.chunk(N)
        assert len(chunks) == N and all(ch.numel() == lay["shard_numel"] for ch in chunks)
        got = oracle.pack(oracle.FLAT_ORIG_TRUE, N, 2, ps.numels(), None, [_bits(v) for v in vals])
        np.testing.assert_array_equal(got, _bits(torch.cat(chunks)))


def test_empty_param_gets_alignment_pad_when_last():
    # reading: every param from the second on starts aligned, even an empty one
    lay = oracle.layout(oracle.FLAT_ORIG_TRUE, 4, 2, [3, 0])
    assert lay["offsets"] == [0, 8] and lay["total_numel"] == 8
    lay = oracle.layout(oracle.FLAT_ORIG_FALSE, 4, 2, [0])
    assert lay["shard_numel"] == 0 and lay["total_numel"] == 0


# ---------------------------------------------------------------------------
# pack / all-gather + unpack round trip
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [oracle.FLAT_ORIG_FALSE, oracle.FLAT_ORIG_TRUE,
                                  oracle.PER_PARAM_DIM0])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N", [3, 5, 7])
def test_all_gather_of_shards_is_original(kind, dtype, N):
    if kind == oracle.PER_PARAM_DIM0:
        ps = W.awkward_2d(N, dtype=dtype)
    else:
        ps = W.awkward_1d(N, kind, dtype)
    eb = 2 if dtype == torch.bfloat16 else 4
    d0, inner = ps.dim0_inner()
    vals = [_bits(v) for v in W.make_params(ps)]
    packed = oracle.pack(kind, N, eb, d0, inner, vals)
    lay = oracle.layout(kind, N, eb, d0, inner)
    # pads are exactly zero: the packed buffer holds every value once and zeros elsewhere
    nonpad = sum(v.size for v in vals)
    assert packed.size == lay["total_numel"]
    if eb == 2:
        assert np.count_nonzero(packed) == sum(np.count_nonzero(v) for v in vals)
    else:
        assert np.count_nonzero(packed.view(np.uint32)) == sum(
            np.count_nonzero(v.view(np.uint32)) for v in vals)
    assert lay["unpadded_numel"] == nonpad
    n_out = 2
    outs = oracle.all_gather_unpack(kind, N, eb, d0, inner, packed, n_out=n_out)
    for rep in outs:
        for got, want in zip(rep, vals):
            np.testing.assert_array_equal(got.view(np.uint8), want.view(np.uint8))


# ---------------------------------------------------------------------------
# reduce-scatter
# ---------------------------------------------------------------------------

def test_reduce_scatter_is_mean_within_fp32_bound():
    rng = np.random.default_rng(5)
    for N in (2, 3, 5, 7, 8):
        c = 257
        bufs = [_bits(torch.from_numpy(rng.normal(0, 1e-2, N * c).astype(np.float32))
                      .to(torch.bfloat16)) for _ in range(N)]
        got = oracle.reduce_scatter(N, c, bufs).astype(np.float64)
        vals = np.stack([oracle.bf16_widen(b).astype(np.float64) for b in bufs])
        exact = vals.sum(axis=0) / N
        bound = (N * 2.0 ** -24) * np.abs(vals).sum(axis=0) / N + 2.0 ** -24 * np.abs(exact)
        assert np.all(np.abs(got - exact) <= bound + 1e-45)


def test_reduce_scatter_exact_when_sums_are_exact():
    # small integers: every partial sum is exact in fp32, so the result is the
    # correctly rounded exact mean
    rng = np.random.default_rng(6)
    for N in (2, 3, 4, 5, 7, 8):
        c = 64
        ints = [rng.integers(-100, 100, N * c) for _ in range(N)]
        bufs = [_bits(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)) for x in ints]
        got = oracle.reduce_scatter(N, c, bufs)
        total = np.sum(np.stack(ints), axis=0).astype(np.float32)
        np.testing.assert_array_equal(got, total / np.float32(N))


def test_reduce_scatter_fixed_rank_order():
    # rank 0: 1.0, ranks 1, 2: 2^-24, rank 3: 0.  In rank order 1 + 2^-24 is a tie that
    # rounds to even (1.0) twice, so the sum is 1 and the mean 0.25 exactly; in reverse
    # order the two small values would first combine to 2^-23 and give 0.25 + 2^-25.
    vals = [1.0, 2.0 ** -24, 2.0 ** -24, 0.0]
    bufs = [_bits(torch.full((4,), v, dtype=torch.float32).to(torch.bfloat16)) for v in vals]
    got = oracle.reduce_scatter(4, 1, bufs)
    assert np.all(got == np.float32(0.25))
    assert np.float32(0.25) != np.float32(0.25 + 2.0 ** -25)


def test_reduce_scatter_all_reduce_identity():
    # all-reduce = reduce-scatter + all-gather: the N shards side by side are the
    # element-wise mean of the whole buffers, whichever rank computed them
    rng = np.random.default_rng(7)
    N, c = 5, 33
    bufs = [rng.normal(0, 1, N * c).astype(np.float32) for _ in range(N)]
    got = oracle.reduce_scatter(N, c, bufs)
    acc = bufs[0].copy()
    for b in bufs[1:]:
        acc = (acc + b).astype(np.float32)
    np.testing.assert_array_equal(got, acc / np.float32(N))


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_cast():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000],
                    dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    x = bits.view(np.float32)
    got = oracle.bf16_round(x)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    # NaN stays a quiet NaN
    g = got[nan].astype(np.uint32)
    assert np.all(((g >> 7) & 0xFF) == 0xFF) and np.all(g & 0x40)
    np.testing.assert_array_equal(oracle.bf16_widen(got[~nan]),
                                  torch.from_numpy(want[~nan].view(np.int16)).view(torch.bfloat16)
                                  .float().numpy())


# ---------------------------------------------------------------------------
# AdamW
# ---------------------------------------------------------------------------

def _torch_adamw_step(theta, m, v, g, hp, step):
    p = torch.nn.Parameter(torch.from_numpy(theta.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                            weight_decay=hp["weight_decay"], foreach=False)
    p.grad = torch.from_numpy(g.astype(np.float64))
    opt.state[p] = {"step": torch.tensor(float(step - 1), dtype=torch.float64),
                    "exp_avg": torch.from_numpy(m.astype(np.float64)),
                    "exp_avg_sq": torch.from_numpy(v.astype(np.float64))}
    opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def _ulps(a32, b32):
    a = a32.astype(np.float32).view(np.int32).astype(np.int64)
    b = b32.astype(np.float32).view(np.int32).astype(np.int64)
    a = np.where(a < 0, -(a & 0x7FFFFFFF), a)
    b = np.where(b < 0, -(b & 0x7FFFFFFF), b)
    return np.abs(a - b)


@pytest.mark.parametrize("wd", [0.0, 0.01, 0.1])
@pytest.mark.parametrize("step", [1, 2, 3, 10, 1000])
def test_adamw_matches_torch_optim(wd, step):
    rng = np.random.default_rng(step * 10 + int(wd * 100))
    n = 4096
    theta = rng.normal(0, 0.02, n).astype(np.float32)
    m = (rng.normal(0, 1e-3, n) if step > 1 else np.zeros(n)).astype(np.float32)
    v = (np.abs(rng.normal(0, 1e-6, n)) if step > 1 else np.zeros(n)).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd)
    t_theta, t_m, t_v = _torch_adamw_step(theta, m, v, g, hp, step)
    mt, mm, vv = theta.copy(), m.copy(), v.copy()
    p = oracle.adamw(g, mt, mm, vv, step=step, **hp)
    assert _ulps(mt, t_theta.astype(np.float32)).max() <= 1
    assert _ulps(mm, t_m.astype(np.float32)).max() <= 1
    assert _ulps(vv, t_v.astype(np.float32)).max() <= 1
    want_p = torch.from_numpy(mt.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(p, want_p)


def test_adamw_first_step_closed_form():
    # t = 1, wd = 0: mhat = g, vhat = g^2, so theta_1 = theta_0 - lr * g / (|g| + eps)
    rng = np.random.default_rng(11)
    n = 1000
    theta = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    z = np.zeros(n, np.float32)
    mt, mm, vv = theta.copy(), z.copy(), z.copy()
    oracle.adamw(g, mt, mm, vv, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                 step=1)
    g64 = g.astype(np.float64)
    closed = theta.astype(np.float64) - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    assert _ulps(mt, closed.astype(np.float32)).max() <= 1
    # moments after one step: (1-b1) g and (1-b2) g^2
    assert _ulps(mm, (0.1 * g64).astype(np.float32)).max() <= 1
    assert _ulps(vv, (0.001 * g64 * g64).astype(np.float32)).max() <= 1


def test_adamw_pad_stays_zero():
    z = np.zeros(64, np.float32)
    mt, mm, vv = z.copy(), z.copy(), z.copy()
    for step in (1, 2, 3):
        p = oracle.adamw(z.copy(), mt, mm, vv, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                         weight_decay=0.01, step=step)
        assert not np.any(mt.view(np.uint32)) and not np.any(mm.view(np.uint32))
        assert not np.any(vv.view(np.uint32)) and not np.any(p)


def test_init_master_widens_every_bf16_pattern_and_zeroes_the_moments():
    """Optimizer-state initialisation ("Scaling data parallel", sections 1 and
    9.1: an fp32 master copy of the bf16 parameters, fp32 Adam moments that
    start at zero), pinned outside the oracle: the master is torch's bf16 ->
    fp32 widening of every one of the 2^16 bf16 bit patterns, NaNs included,
    bit for bit; both moments are +0.0 bit patterns, written over buffers that
    held something else."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = (torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
            .view(np.uint32))
    n = bits.size
    poison = [np.full(n, np.float32(x)) for x in (np.nan, -1.5, 3.0)]
    master, m, v = oracle.init_master(bits, out=poison)
    np.testing.assert_array_equal(master.view(np.uint32), want)
    assert not np.any(m.view(np.uint32)) and not np.any(v.view(np.uint32))


def test_init_master_of_an_fp32_shard_is_the_identity():
    """fp32 plans: the master is the shard itself, bit for bit (any pattern,
    NaNs and signed zeros included), and the moments are +0.0."""
    rng = np.random.default_rng(21)
    x = rng.integers(0, 1 << 32, 1 << 16, dtype=np.uint64).astype(np.uint32)
    x[:4] = [0x00000000, 0x80000000, 0x7F800001, 0xFFC00000]
    shard = x.view(np.float32)
    poison = [np.full(x.size, np.float32(x0)) for x0 in (2.0, np.nan, -7.0)]
    master, m, v = oracle.init_master(shard, out=poison)
    np.testing.assert_array_equal(master.view(np.uint32), x)
    assert not np.any(m.view(np.uint32)) and not np.any(v.view(np.uint32))


# ---------------------------------------------------------------------------
# sharded step == unsharded step (ZeRO changes where state lives, not the math)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind,N", [(oracle.FLAT_ORIG_TRUE, 2), (oracle.FLAT_ORIG_FALSE, 3),
                                    (oracle.PER_PARAM_DIM0, 5)])
def test_sharded_step_equals_unsharded_step(kind, N):
    ps = W.tiny_mlp(N, kind)
    d0, inner = ps.dim0_inner()
    params = [_bits(p) for p in W.make_params(ps)]
    grads = [[_bits(g) for g in rank] for rank in W.make_rank_grads(ps)]
    hp = W.adamw_hparams()
    lay = oracle.layout(kind, N, 2, d0, inner)
    shards = oracle.pack(kind, N, 2, d0, inner, params)
    master, m, v = oracle.init_master(shards)
    packed_grads = [oracle.pack(kind, N, 2, d0, inner, gr) for gr in grads]
    hp1 = {k: hp[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay")}
    new_shards, _ = oracle.reduce_scatter_adamw(N, lay["shard_numel"], packed_grads, master, m, v,
                                                step=1, **hp1)
    full = oracle.all_gather_unpack(kind, N, 2, d0, inner, new_shards)[0]
    # unsharded: per parameter, average the N rank gradients, AdamW the whole tensor
    for i, p in enumerate(params):
        stacked = [grads[r][i] for r in range(N)]
        # a 1-"shard" reduce over N ranks of the whole tensor: pad to N equal pieces
        n = p.size
        c = -(-n // N)
        bufs = [np.concatenate([s, np.zeros(N * c - n, np.uint16)]) for s in stacked]
        mean = oracle.reduce_scatter(N, c, bufs)[:n].copy()
        mt, mm, vv = oracle.init_master(p)
        mt, mm, vv = mt.copy(), mm.copy(), vv.copy()
        newp = oracle.adamw(mean, mt, mm, vv, step=1, **hp1)
        np.testing.assert_array_equal(full[i], newp)


# ---------------------------------------------------------------------------
# DDP buckets
# ---------------------------------------------------------------------------

def test_ddp_bucket_assignment_properties():
    rng = random.Random(9)
    for trial in range(300):
        T = rng.randint(0, 12)
        numels = [rng.randint(0, 50) for _ in range(T)]
        cap = rng.randint(1, 160)
        bucket_of, count = oracle.ddp_buckets(numels, 2, cap)
        order = list(range(T - 1, -1, -1))     # reverse registration order
        # buckets are consecutive runs of the reversed order, numbered 0, 1, ...
        seq = [bucket_of[t] for t in order]
        assert seq == sorted(seq)
        assert (count == 0) == (sum(numels) == 0)
        for b in range(count):
            members = [t for t in order if bucket_of[t] == b]
            size = sum(numels[t] * 2 for t in members)
            last = b == count - 1
            if not last:
                assert size >= cap                          # a closed bucket is full
                assert size - numels[members[-1]] * 2 < cap  # and closed at the first chance
            else:
                assert size > 0          # the open bucket at the end holds something


def test_ddp_bucket_counts_small_cases():
    # 4 tensors of 10 bf16 elements = 20 bytes each
    assert oracle.ddp_buckets([10] * 4, 2, 20)[1] == 4
    assert oracle.ddp_buckets([10] * 4, 2, 40)[1] == 2
    assert oracle.ddp_buckets([10] * 4, 2, 41)[1] == 2   # 60 bytes closes, 20 left open
    assert oracle.ddp_buckets([10] * 4, 2, 1 << 30)[1] == 1
    b, n = oracle.ddp_buckets([1, 2, 3], 2, 6)   # reverse: 3 (6 B) closes alone
    assert b == [1, 1, 0] and n == 2


def test_ddp_average_fixed_rank_order_decides_the_bf16():
    # N = 4, ranks 4, 2^-6, 2^-22, 2^-22 (all exact in bf16).  In rank order the
    # two 2^-22 each meet 4 + 2^-6 at half an fp32 ulp and vanish (ties to even),
    # so the mean is 1 + 2^-8: exactly between the bf16 values 1 and 1 + 2^-7,
    # which rounds to the even one, 1.0 (0x3F80).  Had the small values been
    # added first (reverse order) the mean would be 1 + 2^-8 + 2^-23 and round
    # up to 0x3F81.  The second element holds the ranks reversed, where rank
    # order itself gives the larger sum.
    def b16(x):
        return np.array([np.float32(x)]).view(np.uint32)[0] >> 16
    col0 = [4.0, 2.0 ** -6, 2.0 ** -22, 2.0 ** -22]
    ranks = [[np.array([b16(col0[r]), b16(col0[3 - r])], dtype=np.uint16)] for r in range(4)]
    out = oracle.ddp_average(ranks)[0]
    assert out[0] == 0x3F80
    assert out[1] == 0x3F81


def test_ddp_average_is_rs_mean_rounded():
    rng = np.random.default_rng(12)
    N, T = 8, 5
    numels = [3, 17, 0, 64, 9]
    grads = [[_bits(torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).to(torch.bfloat16))
              for n in numels] for _ in range(N)]
    avg = oracle.ddp_average(grads)
    for t, n in enumerate(numels):
        if n == 0:
            continue
        bufs = [np.concatenate([grads[r][t], np.zeros(N * n - n, np.uint16)]) for r in range(N)]
        rs = oracle.reduce_scatter(N, n, bufs)[:n]
        want = torch.from_numpy(rs.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(avg[t], want)


# ---------------------------------------------------------------------------
# ledger closed forms
# ---------------------------------------------------------------------------

def test_ledger_tables():
    rows = list(_golden_rows("ledger_tables.txt"))
    assert len(rows) >= 19
    for src, scheme, P, N, b, bopt, qty, value, dec in rows:
        P, N, b, bopt = float(P), int(N), float(b), float(bopt)
        if qty == "resident":
            got = ledger.resident_bytes(scheme, P, N, b, bopt)
        elif qty == "worst_peak":
            got = ledger.worst_peak_bytes(scheme, P, N, b, bopt)
        else:
            got = ledger.comm_bytes_per_iter(scheme, P, N, b)
        assert round(got / 1e9, int(dec)) == pytest.approx(float(value)), (src, scheme, qty)


def test_ledger_monotone_in_N():
    # "ai-infra-kb M036" self-check: going from 4 to 8 ranks, only the sharded terms shrink
    for scheme in ("zero1", "zero2", "zero3"):
        assert ledger.resident_bytes(scheme, 7e9, 8, 2, 12) < ledger.resident_bytes(scheme, 7e9, 4, 2, 12)
    assert ledger.resident_bytes("ddp", 7e9, 8, 2, 12) == ledger.resident_bytes("ddp", 7e9, 4, 2, 12)


def test_plan_bytes_at_least_ledger():
    for kind in (oracle.FLAT_ORIG_FALSE, oracle.FLAT_ORIG_TRUE, oracle.PER_PARAM_DIM0):
        for N in (3, 5, 7):
            ps = W.awkward_1d(N, kind, torch.bfloat16)
            lay = oracle.layout(kind, N, 2, ps.numels())
            P = lay["unpadded_numel"]
            planned = ledger.plan_resident_bytes(lay["shard_numel"], 2, 12)
            ideal = ledger.resident_bytes("zero3", P, N, 2, 12)
            assert planned >= ideal
            assert (planned == ideal) == (lay["total_numel"] == P)
    # the 1.2B model divides evenly at N=8: no padding, the ledger is met exactly
    ps = W.llama_1b2()
    d0, inner = ps.dim0_inner()
    total = 0
    lo = 0
    for g in ps.groups:
        total += oracle.layout(oracle.PER_PARAM_DIM0, 8, 2, d0[lo:lo + g], inner[lo:lo + g])["total_numel"]
        lo += g
    assert total == ps.total_unpadded() == 1_364_297_728


# ---------------------------------------------------------------------------
# data parallel == large batch
# ---------------------------------------------------------------------------

def test_dp_mlp_grads_match_autograd_and_fd():
    params, x, t = dp_equivalence.make_problem(B=8)
    loss, grads = dp_equivalence.loss_and_grads(params, x, t)
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in params.items()}
    a = torch.from_numpy(x) @ tp["W_in"] + tp["b_in"]
    o = torch.relu(a) @ tp["W_out"] + tp["b_out"]
    y = torch.nn.functional.layer_norm(o, (o.shape[1],), eps=dp_equivalence.LN_EPS) * tp["ln_w"]
    tl = 0.5 * ((y - torch.from_numpy(t)) ** 2).sum() / x.shape[0]
    tl.backward()
    assert abs(float(tl.detach()) - loss) < 1e-12 * max(1.0, abs(loss))
    for k in grads:
        np.testing.assert_allclose(grads[k], tp[k].grad.numpy(), rtol=1e-10, atol=1e-13)
    # one finite-difference probe per parameter tensor
    for k in params:
        idx = tuple(0 for _ in params[k].shape)
        h = 1e-6
        pp = {kk: vv.copy() for kk, vv in params.items()}
        pp[k][idx] += h
        lp, _ = dp_equivalence.loss_and_grads(pp, x, t)
        pp[k][idx] -= 2 * h
        lm, _ = dp_equivalence.loss_and_grads(pp, x, t)
        assert abs((lp - lm) / (2 * h) - grads[k][idx]) < 1e-6 * max(1.0, abs(grads[k][idx]))


@pytest.mark.parametrize("N", [2, 4, 8])
def test_dp_mean_of_rank_grads_is_large_batch_grad(N):
    params, x, t = dp_equivalence.make_problem(B=16, seed=N)
    _, full = dp_equivalence.loss_and_grads(params, x, t)
    dp = dp_equivalence.rank_mean_grads(params, x, t, [16 // N] * N)
    for k in full:
        rel = np.abs(dp[k] - full[k]).max() / max(np.abs(full[k]).max(), 1e-300)
        assert rel <= 1e-12


def test_dp_unequal_split_needs_token_weighting():
    params, x, t = dp_equivalence.make_problem(B=16, seed=3)
    _, full = dp_equivalence.loss_and_grads(params, x, t)
    plain = dp_equivalence.rank_mean_grads(params, x, t, [2, 14])
    weighted = dp_equivalence.rank_mean_grads(params, x, t, [2, 14], token_weighted=True)
    k = "W_in"
    assert np.abs(plain[k] - full[k]).max() > 1e-6 * np.abs(full[k]).max()
    assert np.abs(weighted[k] - full[k]).max() <= 1e-12 * np.abs(full[k]).max()


# ---------------------------------------------------------------------------
# gradient accumulation
# ---------------------------------------------------------------------------

def test_accumulation_single_micro_batch_is_reduce_scatter():
    rng = np.random.default_rng(21)
    N, c = 5, 77
    bufs = [_bits(torch.from_numpy(rng.normal(0, 1e-2, N * c).astype(np.float32)).to(torch.bfloat16))
            for _ in range(N)]
    acc = oracle.accumulate(N, c, bufs, None)
    np.testing.assert_array_equal(oracle.accumulated_grad(acc, 1), oracle.reduce_scatter(N, c, bufs))


def test_accumulation_identical_micro_batches_average_exactly():
    # acc = RS + RS = 2 RS exactly, and 2 RS / 2 = RS exactly
    rng = np.random.default_rng(22)
    N, c = 8, 64
    bufs = [_bits(torch.from_numpy(rng.normal(0, 1e-3, N * c).astype(np.float32)).to(torch.bfloat16))
            for _ in range(N)]
    acc = oracle.accumulate(N, c, bufs, None)
    acc = oracle.accumulate(N, c, bufs, acc)
    np.testing.assert_array_equal(oracle.accumulated_grad(acc, 2), oracle.reduce_scatter(N, c, bufs))


def test_accumulation_hand_example():
    # N = 2, k = 3 micro-batches, one element per shard (c = 1): rank values
    # micro-batch 1: (1, 3) -> mean 2; 2: (4, 8) -> 6; 3: (-2, 2) -> 0
    # acc = 2 + 6 + 0 = 8, g = 8 / 3 rounded to fp32
    mbs = [(1.0, 3.0), (4.0, 8.0), (-2.0, 2.0)]
    acc = None
    for a, b in mbs:
        bufs = [_bits(torch.tensor([a, a], dtype=torch.float32).to(torch.bfloat16)),
                _bits(torch.tensor([b, b], dtype=torch.float32).to(torch.bfloat16))]
        acc = oracle.accumulate(2, 1, bufs, acc)
    np.testing.assert_array_equal(acc, np.array([8.0, 8.0], np.float32))
    np.testing.assert_array_equal(oracle.accumulated_grad(acc, 3),
                                  np.array([8.0, 8.0], np.float32) / np.float32(3))


@pytest.mark.parametrize("N,k", [(2, 2), (4, 2), (2, 4)])
def test_accumulated_dp_equals_large_batch(N, k):
    params, x, t = dp_equivalence.make_problem(B=16, seed=N * 10 + k)
    _, full = dp_equivalence.loss_and_grads(params, x, t)
    acc = dp_equivalence.accumulated_dp_grads(params, x, t, N, k)
    for key in full:
        rel = np.abs(acc[key] - full[key]).max() / max(np.abs(full[key]).max(), 1e-300)
        assert rel <= 1e-12
