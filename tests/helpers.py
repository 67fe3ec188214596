"""Shared helpers for the tests: tensor <-> numpy bit views and the parity
tolerances used against the oracle."""
from __future__ import annotations

import re
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def to_np(t: torch.Tensor) -> np.ndarray:
    """Any bf16 / fp32 tensor (any device) -> numpy uint16 bits / float32, flattened copy."""
    t = t.detach().reshape(-1).cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    raise TypeError(t.dtype)


def header_functions() -> list:
    """Names of the functions include/shardstate.h declares."""
    with open(os.path.join(ROOT, "include", "shardstate.h")) as f:
        text = f.read()
    body = text[text.index('extern "C" {'):]
    names = re.findall(r"^(?:const\s+)?(?:int|void|uint64_t|const char\*|char\*)\s*\**\s*(\w+)\s*\(", body,
                       re.M)
    return sorted(set(names))


# ---------------------------------------------------------------------------
# tolerances
# ---------------------------------------------------------------------------
# AdamW: the GPU evaluates the update in fp32, the oracle in fp64 rounded once
# to fp32.  Every fp32 operation is within half an ulp, so the difference is
# a few fp32 ulps of the magnitudes of the operands combined:
#   master: |theta_prev| + |theta_new|   (the update is at most their sum)
#   exp_avg: |m_prev| + |g|              (b1*m and (1-b1)*g may cancel)
#   exp_avg_sq: |v_new|                  (two non-negative terms)
# The bound checked is 1e-6 times that magnitude (about eight ulps).
# bf16 parameters: the round-to-nearest-even of masters that differ by a few
# fp32 ulps can differ by at most one bf16 ulp.
RTOL = 1e-6

# How much of the tolerance each check used, one record per call, printed by
# the terminal summary in conftest.py: per array the largest error relative to
# the oracle's result, and how many elements lie beyond a strict 1e-6 of the
# result (the bound the operand-relative one replaces where terms cancel) or
# beyond one bf16 ulp.
MARGINS = []


def _case() -> str:
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def _result_relative(gpu, ref):
    """|gpu - ref| / |ref| per element (0 where both are equal, inf where ref
    is 0 and gpu is not)."""
    d = np.abs(gpu - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d == 0, 0.0, d / np.abs(ref))
    return np.nan_to_num(r, nan=np.inf)


def _record(kind, n, **fields):
    MARGINS.append(dict(case=_case(), kind=kind, n=int(n), **fields))


def check_adamw_state(gpu_master, gpu_m, gpu_v, ref_master, ref_m, ref_v, prev_master, prev_m,
                      grad):
    gm = np.asarray(gpu_master, np.float64)
    rm = np.asarray(ref_master, np.float64)
    rel = {name: _result_relative(np.asarray(g, np.float64), np.asarray(r, np.float64))
           for name, g, r in (("master", gpu_master, ref_master), ("exp_avg", gpu_m, ref_m),
                              ("exp_avg_sq", gpu_v, ref_v))}
    _record("state", gm.size,
            **{f"max_rel_{k}": float(v.max(initial=0.0)) for k, v in rel.items()},
            **{f"n_beyond_1e-6_{k}": int((v > RTOL).sum()) for k, v in rel.items()})
    scale = np.abs(np.asarray(prev_master, np.float64)) + np.abs(rm)
    bad = np.abs(gm - rm) > RTOL * scale
    assert not bad.any(), f"master: {bad.sum()} elements beyond tolerance, first at {np.argmax(bad)}"
    gmm = np.asarray(gpu_m, np.float64)
    rmm = np.asarray(ref_m, np.float64)
    scale = np.abs(np.asarray(prev_m, np.float64)) + np.abs(np.asarray(grad, np.float64))
    bad = np.abs(gmm - rmm) > RTOL * scale
    assert not bad.any(), f"exp_avg: {bad.sum()} elements beyond tolerance"
    gv = np.asarray(gpu_v, np.float64)
    rv = np.asarray(ref_v, np.float64)
    bad = np.abs(gv - rv) > RTOL * np.abs(rv)
    assert not bad.any(), f"exp_avg_sq: {bad.sum()} elements beyond tolerance"


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between bit patterns (sign-magnitude -> ordered ints)."""
    def ordered(x):
        x = x.astype(np.int64)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def check_bf16_within_one_ulp(gpu, ref):
    d = bf16_ulp_distance(np.asarray(gpu, np.uint16), np.asarray(ref, np.uint16))
    assert d.max(initial=0) <= 1, f"bf16 params: max distance {d.max()} ulp"


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 2.0 ** -126)))
    return 2.0 ** (np.maximum(e, -126) - 7)


def check_bf16_params(gpu_bits, ref_bits, gpu_master, ref_master, prev_master):
    """bf16 parameter shards against the oracle.
    (a) exact: every bf16 value is the round-to-nearest-even of the GPU's own
        fp32 master (the cast itself is checked bit for bit with the oracle's
        rounding routine);
    (b) within one bf16 ulp of the oracle's parameter -- except where the
        decayed weight and the Adam update nearly cancel: there the fp32
        masters may legitimately differ by the master tolerance (RTOL times
        |theta_prev| + |theta_new|), which can exceed a bf16 ulp of the small
        result, so the bound is one bf16 ulp plus that tolerance.
    Returns the number of elements that needed the widened bound."""
    import oracle
    gpu_bits = np.asarray(gpu_bits, np.uint16)
    np.testing.assert_array_equal(gpu_bits, oracle.bf16_round(np.asarray(gpu_master, np.float32)))
    return check_bf16_close(gpu_bits, ref_bits, ref_master, prev_master)


def check_bf16_close(gpu_bits, ref_bits, ref_master, prev_master):
    """Part (b) of check_bf16_params alone (for the recipe without an fp32
    master, where the GPU keeps no fp32 value to compare the cast against)."""
    import oracle
    gpu_bits = np.asarray(gpu_bits, np.uint16)
    d = bf16_ulp_distance(gpu_bits, np.asarray(ref_bits, np.uint16))
    far = d > 1
    _record("bf16", d.size, max_ulp=int(d.max(initial=0)), n_beyond_1_ulp=int(far.sum()),
            n_off_by_1_ulp=int((d == 1).sum()))
    if not far.any():
        return 0
    rm = np.asarray(ref_master, np.float64)[far]
    tol = RTOL * (np.abs(np.asarray(prev_master, np.float64)[far]) + np.abs(rm))
    gv = oracle.bf16_widen(gpu_bits[far]).astype(np.float64)
    bad = np.abs(gv - rm) > _bf16_ulp(rm) + tol
    assert not bad.any(), (f"bf16 params: {bad.sum()} elements beyond one ulp + master tolerance; "
                           f"first gpu={gv[bad][0]!r} oracle master={rm[bad][0]!r}")
    return int(far.sum())
