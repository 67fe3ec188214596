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


def from_np(a: np.ndarray, device="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32).copy()).to(device)


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


def check_adamw_state(gpu_master, gpu_m, gpu_v, ref_master, ref_m, ref_v, prev_master, prev_m,
                      grad):
    gm = np.asarray(gpu_master, np.float64)
    rm = np.asarray(ref_master, np.float64)
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
