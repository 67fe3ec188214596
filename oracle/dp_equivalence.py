"""Data parallelism equals large-batch training: fp64 gradients of a tiny MLP.

TEST INFRASTRUCTURE (part of the oracle; see ``oracle/__init__.py``).

"Scaling data parallel", section 2.2: with a mean loss over B samples split
evenly across N ranks, each rank's local loss is the mean over its B/N
samples, and the average of the N local gradients equals the full-batch
gradient exactly; with unequal per-rank sizes the ranks must be weighted by
their sample (token) counts.  Section 2.3 writes the model as W_in[D,F] and
W_out[F,D]; the pages give no activation or norm, so this module takes
  a = x W_in + b_in,  h = relu(a),  o = h W_out + b_out,
  y = LayerNorm(o) * w_ln  (no bias, eps 1e-5),
  loss = mean over samples of 0.5 * ||y - t||^2,
with the backward pass written out by hand in numpy float64.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np

LN_EPS = 1e-5
PARAM_NAMES = ("W_in", "b_in", "W_out", "b_out", "ln_w")


def loss_and_grads(params: Dict[str, np.ndarray], x: np.ndarray, t: np.ndarray):
    """Mean loss over the rows of x and its gradient w.r.t. every parameter."""
    W_in, b_in = params["W_in"], params["b_in"]
    W_out, b_out, w_ln = params["W_out"], params["b_out"], params["ln_w"]
    B = x.shape[0]
    a = x @ W_in + b_in
    h = np.maximum(a, 0.0)
    o = h @ W_out + b_out
    mu = o.mean(axis=1, keepdims=True)
    var = ((o - mu) ** 2).mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + LN_EPS)
    xhat = (o - mu) * rstd
    y = xhat * w_ln
    diff = y - t
    loss = 0.5 * (diff ** 2).sum() / B

    dy = diff / B
    d_ln = (dy * xhat).sum(axis=0)
    dxhat = dy * w_ln
    do = rstd * (dxhat - dxhat.mean(axis=1, keepdims=True)
                 - xhat * (dxhat * xhat).mean(axis=1, keepdims=True))
    dW_out = h.T @ do
    db_out = do.sum(axis=0)
    dh = do @ W_out.T
    da = dh * (a > 0)
    dW_in = x.T @ da
    db_in = da.sum(axis=0)
    return loss, {"W_in": dW_in, "b_in": db_in, "W_out": dW_out, "b_out": db_out, "ln_w": d_ln}


def rank_mean_grads(params, x, t, splits: Sequence[int], token_weighted: bool = False):
    """Average of per-rank gradients, ranks holding consecutive row blocks of
    the given sizes.  token_weighted weights rank r by splits[r] / B."""
    B = x.shape[0]
    assert sum(splits) == B
    acc = {k: np.zeros_like(v) for k, v in params.items()}
    lo = 0
    N = len(splits)
    for n_r in splits:
        _, g = loss_and_grads(params, x[lo:lo + n_r], t[lo:lo + n_r])
        w = (n_r / B) if token_weighted else (1.0 / N)
        for k in acc:
            acc[k] += w * g[k]
        lo += n_r
    return acc


def accumulated_dp_grads(params, x, t, world_size: int, micro_batches: int):
    """Gradient accumulation on top of data parallelism: the batch is split into
    `micro_batches` consecutive micro-batches, each split evenly over
    `world_size` ranks; the step's gradient is the mean over micro-batches of
    the rank-mean gradients ("Scaling data parallel", sections 2.2 and 5:
    data parallelism is gradient accumulation done in parallel)."""
    B = x.shape[0]
    mb = B // micro_batches
    acc = {k: np.zeros_like(v) for k, v in params.items()}
    for j in range(micro_batches):
        xs, ts = x[j * mb:(j + 1) * mb], t[j * mb:(j + 1) * mb]
        g = rank_mean_grads(params, xs, ts, [mb // world_size] * world_size)
        for k in acc:
            acc[k] += g[k] / micro_batches
    return acc


def make_problem(D: int = 64, F: int = 128, B: int = 16, seed: int = 0):
    rng = np.random.default_rng(seed)
    params = {
        "W_in": rng.normal(0, 0.02 * 8, (D, F)),
        "b_in": rng.normal(0, 0.02, (F,)),
        "W_out": rng.normal(0, 0.02 * 8, (F, D)),
        "b_out": rng.normal(0, 0.02, (D,)),
        "ln_w": 1.0 + rng.normal(0, 0.02, (D,)),
    }
    x = rng.normal(0, 1, (B, D))
    t = rng.normal(0, 1, (B, D))
    return params, x, t
