"""Set-up shared by the GPU parity tests: a plan plus device buffers for a
parameter set, and the oracle's answers for the same inputs (group by group,
since the oracle plans one group at a time)."""
from __future__ import annotations

from typing import List

import numpy as np
import torch

import oracle
import workloads as W
from tests.helpers import to_np

GUARD = 64  # guard-band elements before and after every output buffer
SENTINEL_BF16 = 0x7FBF  # a NaN pattern nothing in the path produces
SENTINEL_F32 = float.fromhex("0x1.5555p+100")


def guarded(numel: int, dtype: torch.dtype, device="cuda"):
    """A tensor of `numel` elements with sentinel guard bands on both sides;
    returns (interior view, whole buffer).  16-byte alignment is kept."""
    whole = torch.empty(numel + 2 * GUARD, dtype=dtype, device=device)
    if dtype == torch.bfloat16:
        whole.view(torch.int16).fill_(SENTINEL_BF16)
    else:
        whole.fill_(SENTINEL_F32)
    return whole[GUARD:GUARD + numel], whole


def guards_intact(whole: torch.Tensor) -> bool:
    g = torch.cat([whole[:GUARD], whole[-GUARD:]])
    if g.dtype == torch.bfloat16:
        return bool((g.view(torch.int16) == SENTINEL_BF16).all())
    return bool((g == SENTINEL_F32).all())


def elem_bytes(dtype) -> int:
    return 2 if dtype == torch.bfloat16 else 4


class Setup:
    """Plan + params for a ParamSet, and oracle helpers working group by group."""

    def __init__(self, ss, ps: W.ParamSet, device="cuda", make_values=True):
        self.ss = ss
        self.ps = ps
        self.kind = ps.layout
        self.N = ps.world_size
        self.eb = elem_bytes(ps.dtype)
        self.d0, self.inner = ps.dim0_inner()
        self.plan = ss.fsdp_plan_create(self.kind, self.N, self.eb, self.d0, self.inner,
                                        group_num_params=ps.groups)
        self.info = self.plan.info()
        self.total = self.info.total_numel
        self.groups = [ss.fsdp_plan_group(self.plan, g) for g in range(len(ps.groups))]
        if make_values:
            self.params_cpu = W.make_params(ps)
            self.params = [p.to(device) for p in self.params_cpu]

    # oracle, group by group ------------------------------------------------
    def _group_args(self, g):
        grp = self.groups[g]
        a, b = grp["first_param"], grp["first_param"] + grp["num_params"]
        return a, b, self.d0[a:b], self.inner[a:b]

    def oracle_pack(self, arrays: List[np.ndarray]) -> np.ndarray:
        out = []
        for g in range(len(self.groups)):
            a, b, d0, inner = self._group_args(g)
            out.append(oracle.pack(self.kind, self.N, self.eb, d0, inner, arrays[a:b]))
        return np.concatenate(out) if out else np.zeros(0, np.uint16 if self.eb == 2 else np.float32)

    def oracle_unpack(self, shards: np.ndarray, n_out: int = 1):
        reps = [[] for _ in range(n_out)]
        for g in range(len(self.groups)):
            a, b, d0, inner = self._group_args(g)
            base = self.groups[g]["base"]
            span = self.N * self.groups[g]["shard_numel"]
            outs = oracle.all_gather_unpack(self.kind, self.N, self.eb, d0, inner,
                                            shards[base:base + span], n_out=n_out)
            for j in range(n_out):
                reps[j].extend(outs[j])
        return reps

    def params_np(self):
        return [to_np(p) for p in self.params_cpu]
