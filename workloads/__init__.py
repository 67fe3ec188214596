"""Seeded synthetic workloads for the sharded-state step.

This module holds shapes and random numbers only: it does none of the
method's arithmetic (no layout, no reduction, no optimizer).  Both the CUDA
path's tests/bench and the CPU oracle draw their inputs from here, so the two
sides see identical bytes.

Shapes follow the model families the pages use as workloads:
  * a tiny two-matrix MLP (the W_in[D,F] / W_out[F,D] block of
    "Scaling data parallel", section 2.3) plus a LayerNorm weight;
  * one Llama-style transformer block at hidden 4096;
  * awkward 1-D / 2-D parameter lists whose sizes do not divide N, so
    FlatParameter chunk boundaries split parameters
    ("FSDP1 vs FSDP2", section 03 and the 3+5-element example table);
  * a DDP gradient list of many LayerNorm-sized and a few large tensors
    ("Scaling data parallel", section 4, gradient bucketing);
  * a 1.2B Llama-shaped model wrapped as one fully_shard group per block plus
    a root group ("ai-infra-kb M036", section 04 usage snippet).

Values: parameters N(0, 0.02), gradients N(0, sigma), awkward sets U(-1, 1);
all drawn in fp32 from a seeded torch generator and then rounded to the
storage dtype by torch's own cast.
"""
from __future__ import annotations

import dataclasses
import random
from typing import List, Optional, Sequence, Tuple

import torch

# layout kinds (numbering mirrors the C ABI enum)
FLAT_ORIG_FALSE = 0
FLAT_ORIG_TRUE = 1
PER_PARAM_DIM0 = 2

LAYOUT_NAMES = {FLAT_ORIG_FALSE: "flat_orig_false", FLAT_ORIG_TRUE: "flat_orig_true",
                PER_PARAM_DIM0: "per_param_dim0"}


@dataclasses.dataclass
class ParamSet:
    """An ordered list of named parameter shapes, split into fully_shard groups."""
    names: List[str]
    shapes: List[Tuple[int, ...]]
    groups: List[int]            # number of params in each group, in order
    world_size: int
    layout: int
    dtype: torch.dtype
    seed: int
    param_std: float = 0.02
    grad_std: float = 1e-3
    uniform: bool = False        # U(-1,1) instead of normal values
    description: str = ""

    @property
    def num_params(self) -> int:
        return len(self.shapes)

    def numels(self) -> List[int]:
        out = []
        for s in self.shapes:
            n = 1
            for d in s:
                n *= d
            out.append(n)
        return out

    def dim0_inner(self) -> Tuple[List[int], List[int]]:
        """dim-0 size and elements per dim-0 row; a 0-d shape counts as [1]."""
        d0, inner = [], []
        for s in self.shapes:
            if len(s) == 0:
                d0.append(1)
                inner.append(1)
                continue
            d0.append(s[0])
            r = 1
            for d in s[1:]:
                r *= d
            inner.append(r)
        return d0, inner

    def total_unpadded(self) -> int:
        return sum(self.numels())


# ----------------------------------------------------------------------------
# config shapes
# ----------------------------------------------------------------------------

def tiny_mlp(world_size: int = 2, layout: int = FLAT_ORIG_TRUE) -> ParamSet:
    """Two-matrix MLP with biases and a LayerNorm weight, D=64, F=128."""
    names = ["W_in", "b_in", "W_out", "b_out", "ln_w"]
    shapes = [(64, 128), (128,), (128, 64), (64,), (64,)]
    return ParamSet(names, shapes, [len(shapes)], world_size, layout, torch.bfloat16,
                    seed=0, param_std=0.02, grad_std=1e-2,
                    description="tiny 2-layer MLP, 16,640 params")


def _llama_block(prefix: str, hidden: int, ffn: int):
    names = [f"{prefix}q_proj", f"{prefix}k_proj", f"{prefix}v_proj", f"{prefix}o_proj",
             f"{prefix}gate_proj", f"{prefix}up_proj", f"{prefix}down_proj",
             f"{prefix}input_norm", f"{prefix}post_attn_norm"]
    shapes = [(hidden, hidden)] * 4 + [(ffn, hidden), (ffn, hidden), (hidden, ffn),
                                       (hidden,), (hidden,)]
    return names, shapes


def llama_block_4096(world_size: int = 8) -> ParamSet:
    """One Llama-style block at hidden 4096, FFN 11008 (MHA), 202,383,360 params."""
    names, shapes = _llama_block("", 4096, 11008)
    return ParamSet(names, shapes, [len(shapes)], world_size, PER_PARAM_DIM0, torch.bfloat16,
                    seed=1, param_std=0.02, grad_std=1e-3,
                    description="one Llama-style block, hidden 4096, FFN 11008")


def llama_1b2(world_size: int = 8, layers: int = 24, hidden: int = 2048, ffn: int = 5632,
              vocab: int = 32000) -> ParamSet:
    """1.2B Llama-shaped model: one group per block, then a root group holding the
    untied embedding, the final RMSNorm and the LM head (1,364,297,728 params)."""
    names: List[str] = []
    shapes: List[Tuple[int, ...]] = []
    groups: List[int] = []
    for l in range(layers):
        n, s = _llama_block(f"layers.{l}.", hidden, ffn)
        names += n
        shapes += s
        groups.append(len(s))
    names += ["embed_tokens", "norm", "lm_head"]
    shapes += [(vocab, hidden), (hidden,), (vocab, hidden)]
    groups.append(3)
    return ParamSet(names, shapes, groups, world_size, PER_PARAM_DIM0, torch.bfloat16,
                    seed=4, param_std=0.02, grad_std=1e-3,
                    description=f"{layers}-layer Llama-shaped model, hidden {hidden}, "
                                f"FFN {ffn}, vocab {vocab}, {layers} block groups + root")


def awkward_1d(world_size: int, layout: int, dtype: torch.dtype, count: int = 200,
               max_len: int = 5000, seed: int = 2) -> ParamSet:
    """`count` 1-D params with lengths uniform in [0, max_len]; empties forced at
    index 0, count//2 and count-1.  Values U(-1, 1)."""
    rng = random.Random(seed)
    lens = [rng.randint(0, max_len) for _ in range(count)]
    for i in (0, count // 2, count - 1):
        lens[i] = 0
    shapes = [(n,) for n in lens]
    names = [f"p{i}" for i in range(count)]
    return ParamSet(names, shapes, [count], world_size, layout, dtype, seed=seed,
                    uniform=True, description=f"{count} awkward 1-D params")


def awkward_2d(world_size: int, dtype: torch.dtype = torch.bfloat16, count: int = 200,
               max_rows: int = 5000, seed: int = 2) -> ParamSet:
    """`count` 2-D params [d0, inner] with d0 uniform in [0, max_rows] and inner in {1,3,8}."""
    rng = random.Random(seed + 1000)
    shapes = []
    for i in range(count):
        d0 = rng.randint(0, max_rows)
        inner = rng.choice([1, 3, 8])
        shapes.append((d0, inner))
    for i in (0, count // 2, count - 1):
        shapes[i] = (0, shapes[i][1])
    names = [f"p{i}" for i in range(count)]
    return ParamSet(names, shapes, [count], world_size, PER_PARAM_DIM0, dtype, seed=seed,
                    uniform=True, description=f"{count} awkward 2-D params")


@dataclasses.dataclass
class DDPSet:
    numels: List[int]
    world_size: int
    seed: int
    grad_std: float = 1e-3
    description: str = ""


def ddp_grads(world_size: int = 8, n_small: int = 1400, small: int = 2048, n_large: int = 600,
              large: int = 4194304, seed: int = 3) -> DDPSet:
    """DDP gradient list: LayerNorm-sized and large tensors in a seeded random order."""
    numels = [small] * n_small + [large] * n_large
    random.Random(seed).shuffle(numels)
    return DDPSet(numels, world_size, seed,
                  description=f"{n_small}x{small} + {n_large}x{large} bf16 grads")


DDP_BUCKET_CAPS = [64 << 10, 256 << 10, 1 << 20, 4 << 20, 16 << 20, 25 << 20, 64 << 20,
                   256 << 20, 1 << 30]


# ----------------------------------------------------------------------------
# value generators
# ----------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _fill(numel: int, std: float, uniform: bool, dtype: torch.dtype, g: torch.Generator,
          device) -> torch.Tensor:
    if uniform:
        x = torch.rand(numel, generator=g, device=device, dtype=torch.float32) * 2.0 - 1.0
    else:
        x = torch.randn(numel, generator=g, device=device, dtype=torch.float32) * std
    return x.to(dtype)


def make_params(ps: ParamSet, device="cpu") -> List[torch.Tensor]:
    """Per-parameter tensors (contiguous, the set's dtype)."""
    g = _gen(ps.seed, device)
    out = []
    for shape, n in zip(ps.shapes, ps.numels()):
        out.append(_fill(n, ps.param_std, ps.uniform, ps.dtype, g, device).reshape(shape))
    return out


def make_rank_grads(ps: ParamSet, device="cpu") -> List[List[torch.Tensor]]:
    """For each virtual rank, per-parameter gradient tensors (unsharded, unpacked)."""
    g = _gen(ps.seed * 7919 + 17, device)
    out = []
    for _ in range(ps.world_size):
        out.append([_fill(n, ps.grad_std, ps.uniform, ps.dtype, g, device).reshape(s)
                    for s, n in zip(ps.shapes, ps.numels())])
    return out


def make_packed_rank_grads(world_size: int, total_numel: int, std: float, seed: int,
                           dtype=torch.bfloat16, device="cpu",
                           pad_mask: Optional[torch.Tensor] = None) -> List[torch.Tensor]:
    """N flat gradient buffers already in packed (rank-major) layout.  Where a
    pad mask (True = pad) is given, those entries are zero, as a packing step
    leaves them.  Used at sizes where drawing per-parameter tensors first would
    only cost time."""
    g = _gen(seed * 7919 + 17, device)
    out = []
    for _ in range(world_size):
        x = _fill(total_numel, std, False, dtype, g, device)
        if pad_mask is not None:
            x[pad_mask] = 0
        out.append(x)
    return out


def make_ddp_grads(ds: DDPSet, device="cpu", dtype=torch.bfloat16) -> List[List[torch.Tensor]]:
    g = _gen(ds.seed, device)
    return [[_fill(n, ds.grad_std, False, dtype, g, device) for n in ds.numels]
            for _ in range(ds.world_size)]


def adamw_hparams(step: int = 1):
    """AdamW hyper-parameters used for every config (tiny-MLP config values)."""
    return dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=step)


def describe(ps: ParamSet) -> dict:
    return {"description": ps.description, "params": ps.total_unpadded(),
            "num_tensors": ps.num_params, "groups": len(ps.groups),
            "world_size": ps.world_size, "layout": LAYOUT_NAMES[ps.layout],
            "dtype": str(ps.dtype).replace("torch.", ""), "seed": ps.seed}
