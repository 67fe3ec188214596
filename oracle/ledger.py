"""Closed-form memory and communication ledgers of DP / ZeRO / FSDP.

TEST INFRASTRUCTURE (part of the oracle; see ``oracle/__init__.py``).

Notation: P parameters, N data-parallel ranks, b bytes per parameter and per
gradient element, bopt optimizer-state bytes per parameter.

* Resident bytes per rank, "FSDP1 vs FSDP2" ZeRO table (section 02):
  DDP P(2b+bopt); ZeRO-1 2Pb + P bopt/N; ZeRO-2 Pb + P(b+bopt)/N;
  ZeRO-3 / FULL_SHARD P(2b+bopt)/N.  The same four rows appear in
  "Scaling data parallel" section 9 with b = 2 and bopt = k.
* Worst peak ("FSDP1 vs FSDP2", ledger caption): resident plus one full
  parameter copy for FULL_SHARD and SHARD_GRAD_OP; NO_SHARD has no extra copy.
* Communication per iteration per rank ("FSDP1 vs FSDP2", strategy table):
  FULL_SHARD 3P(N-1)/N elements (forward all-gather, backward all-gather,
  backward reduce-scatter); SHARD_GRAD_OP and NO_SHARD 2P(N-1)/N.
"""
from __future__ import annotations


def resident_bytes(scheme: str, P: float, N: int, b: float, bopt: float) -> float:
    s = scheme.lower()
    if s in ("ddp", "dp", "no_shard"):
        return P * (2 * b + bopt)
    if s == "zero1":
        return 2 * P * b + P * bopt / N
    if s == "zero2":
        return P * b + P * (b + bopt) / N
    if s in ("zero3", "full_shard", "shard_grad_op"):
        return P * (2 * b + bopt) / N
    raise ValueError(scheme)


def worst_peak_bytes(scheme: str, P: float, N: int, b: float, bopt: float) -> float:
    s = scheme.lower()
    resident = resident_bytes(s, P, N, b, bopt)
    if s in ("full_shard", "shard_grad_op", "zero3"):
        return resident + P * b
    if s in ("no_shard", "ddp", "dp"):
        return resident
    raise ValueError(scheme)


def comm_elements_per_iter(scheme: str, P: float, N: int) -> float:
    s = scheme.lower()
    if s in ("full_shard", "zero3"):
        return 3 * P * (N - 1) / N
    if s in ("shard_grad_op", "no_shard", "ddp", "zero1", "zero2"):
        return 2 * P * (N - 1) / N
    raise ValueError(scheme)


def comm_bytes_per_iter(scheme: str, P: float, N: int, b: float) -> float:
    return comm_elements_per_iter(scheme, P, N) * b


def plan_resident_bytes(shard_numel: int, b: float, bopt: float) -> float:
    """Per-rank resident bytes of an actual padded plan: every rank stores its
    shard of parameters, gradients and optimizer state."""
    return shard_numel * (2 * b + bopt)
