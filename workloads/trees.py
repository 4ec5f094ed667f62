"""Seeded token trees for tree verification.  Holds no step of the method:
shapes, logits, proposals drawn from the draft distributions, uniforms."""
from __future__ import annotations

import numpy as np

from .configs import STREAM_DRAFT, STREAM_UNIFORMS, _gumbel_rows, as_f32, categorical_draws, quantize
from .philox import uniform_grid


def full_tree(arity: int, depth: int) -> np.ndarray:
    """Parents of a full `arity`-ary tree with `depth` levels below the root,
    nodes numbered breadth first (parent[n] < n; parent[0] = -1)."""
    parent = [-1]
    level = [0]
    for _ in range(depth):
        nxt = []
        for v in level:
            for _ in range(arity):
                parent.append(v)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.asarray(parent, np.int32)


def _children(parent: np.ndarray, v: int) -> list[int]:
    return [n for n in range(len(parent)) if parent[n] == v]


def make_tree_host(B: int, parent, V: int, dtype: str, sigma_t: float, sigma_d: float,
                   temps, seed: int) -> dict:
    """B trees of one shape.  Row n of the target / draft logits is the
    distribution after node n: target N(0, sigma_t^2), draft = target +
    N(0, sigma_d^2), rounded to dtype.  The children of node v are drawn
    independently from softmax(draft_v / T) (Gumbel-max), or at T = 0 are the
    draft's top tokens in rank order.  uniforms[:, 0] is the final draw."""
    parent = np.asarray(parent, np.int32)
    N = len(parent)
    temps = np.asarray(temps, np.float32) if not np.isscalar(temps) else np.full(B, float(temps), np.float32)
    rng = np.random.Generator(np.random.PCG64(seed))
    t32 = rng.standard_normal((B, N, V), dtype=np.float32) * np.float32(sigma_t)
    tgt = quantize(t32, dtype)
    tq = as_f32(tgt, dtype)
    noise = rng.standard_normal((B, N, V), dtype=np.float32) * np.float32(sigma_d)
    drf = quantize(tq + noise, dtype)
    dq = as_f32(drf, dtype).astype(np.float64)
    g = _gumbel_rows(seed + 17, B * N, V).reshape(B, N, V)
    T = temps.astype(np.float64).reshape(B, 1)
    tok = np.zeros((B, N), np.int32)
    for v in range(N):
        kids = _children(parent, v)
        if not kids:
            continue
        order = np.argsort(-dq[:, v], axis=-1, kind="stable")
        for rank, n in enumerate(kids):
            samp = np.argmax(dq[:, v] / np.where(T > 0, T, 1.0) + g[:, n], axis=-1)
            tok[:, n] = np.where(T[:, 0] > 0, samp, order[:, min(rank, V - 1)])
    uni = uniform_grid(seed, STREAM_UNIFORMS, B, N)
    return dict(target=tgt, draft=drf, dtype=dtype, tokens=tok, parent=np.tile(parent, (B, 1)),
                uniforms=uni, temperature=temps, n_nodes=np.full(B, N, np.int32), B=B, N=N, V=V)


def make_tree_pair(p, q, B: int, arity: int, seed: int) -> dict:
    """A root with `arity` children drawn independently from q (Philox
    uniforms, inverse CDF), target row log p and draft row log q at the root;
    the leaves' rows are log p.  fp32, T = 1."""
    p = np.asarray(p, np.float64)
    q = np.asarray(q, np.float64)
    V = len(p)
    N = 1 + arity
    with np.errstate(divide="ignore"):
        lp = np.log(p).astype(np.float32)
        lq = np.log(q).astype(np.float32)
    tgt = np.empty((B, N, V), np.float32)
    tgt[:] = lp
    drf = np.empty((B, N, V), np.float32)
    drf[:] = lq
    ud = uniform_grid(seed, STREAM_DRAFT, B, N)
    tok = np.zeros((B, N), np.int32)
    tok[:, 1:] = categorical_draws(q, ud[:, 1:].reshape(-1)).reshape(B, arity)
    parent = np.zeros(N, np.int32)
    parent[0] = -1
    uni = uniform_grid(seed, STREAM_UNIFORMS, B, N)
    return dict(target=tgt, draft=drf, dtype="f32", tokens=tok, parent=np.tile(parent, (B, 1)),
                uniforms=uni, temperature=np.ones(B, np.float32), n_nodes=np.full(B, N, np.int32),
                B=B, N=N, V=V)
